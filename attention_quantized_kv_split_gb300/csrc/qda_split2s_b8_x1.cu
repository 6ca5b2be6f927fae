// Lean split-kernel instantiations for 8-bit codes, fp32 outputs (exact V codes), D = 64 and 128.
#include "qda_split2.cuh"

cudaError_t qda_launch_split2s_b8_x1(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem,
                                         cudaStream_t s) {
  return qda::launch_split2<8, true, 0>(p, D, nh, ng, grid, smem, s);
}

cudaError_t qda_occupancy_split2s_b8_x1(int D, int nh, int ng, size_t smem, int* n) {
  return qda::occupancy_split2<8, true, 0>(D, nh, ng, smem, n);
}
