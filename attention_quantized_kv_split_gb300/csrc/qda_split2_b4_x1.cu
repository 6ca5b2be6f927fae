// Lean split-kernel instantiations for 4-bit codes, fp32 outputs (exact V codes): D = 256 and 512 here, D = 64 and 128 in
// qda_split2s_b4_x1.cu.
#include "qda_split2.cuh"

cudaError_t qda_launch_split2_b4_x1(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem,
                                        cudaStream_t s) {
  if (D <= 128) return qda_launch_split2s_b4_x1(p, D, nh, ng, grid, smem, s);
  return qda::launch_split2<4, true, 1>(p, D, nh, ng, grid, smem, s);
}

cudaError_t qda_occupancy_split2_b4_x1(int D, int nh, int ng, size_t smem, int* n) {
  if (D <= 128) return qda_occupancy_split2s_b4_x1(D, nh, ng, smem, n);
  return qda::occupancy_split2<4, true, 1>(D, nh, ng, smem, n);
}
