// Tensor-core split-kernel instantiations, 16-bit outputs (V codes as 0.5 + c / 256).
#include "qda_tc.cuh"

cudaError_t qda_launch_tc_x0(const QdaParams& p, const void* tmap_k, int D, int nh, int ng, dim3 grid, size_t smem,
                            cudaStream_t s) {
  return qda::with_tc_kernel<false>(D, nh, ng, p.f16 != 0, [&](auto kern) -> cudaError_t {
    cudaError_t e = qda::ensure_smem_limit(kern, smem);
    if (e != cudaSuccess) return e;
    return qda::launch_pdl(kern, grid, QDA_TC_THREADS, smem, s, true, p, *static_cast<const CUtensorMap*>(tmap_k));
  });
}

cudaError_t qda_occupancy_tc_x0(int D, int nh, int ng, size_t smem, int* n) {
  // the fp16 and bf16 instances have the same resources (one CTA per SM)
  return qda::with_tc_kernel<false>(D, nh, ng, false, [&](auto kern) -> cudaError_t {
    cudaError_t e = qda::ensure_smem_limit(kern, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, QDA_TC_THREADS, smem);
  });
}
