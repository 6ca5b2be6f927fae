// General split-kernel instantiations for 4-bit codes.
#include "qda_split.cuh"

cudaError_t qda_launch_split1_b4(const QdaParams& p, int wpl, int lpr, int nh, dim3 grid, size_t smem, cudaStream_t s) {
  return qda::launch_split<4>(p, wpl, lpr, nh, grid, smem, s);
}

cudaError_t qda_occupancy_split1_b4(int wpl, int lpr, int nh, size_t smem, int* n) {
  return qda::occupancy_split<4>(wpl, lpr, nh, smem, n);
}
