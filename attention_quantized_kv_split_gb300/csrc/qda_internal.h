// Internal definitions shared by the host entry points and the sm_103a kernels of libqdecode_attn.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "qdecode_attn.h"

#define QDA_NW 4                         // consumer warps per CTA of the split kernel
#define QDA_THREADS ((QDA_NW + 1) * 32)  // + one producer warp that drives the bulk copies
#define QDA_SPLIT2_TILE 64                // rows per pipeline stage of the lean split kernel

// Launch parameters of the split and merge kernels (passed by value as a __grid_constant__).
struct QdaParams {
  const void* q;              // [B, L, H, D] input dtype
  const uint32_t* kp;         // packed K codes, rows of W words
  const uint16_t* ks;         // K scales, rows of NG 16-bit values
  const uint16_t* kb;         // K biases
  const uint32_t* vp;
  const uint16_t* vs;
  const uint16_t* vb;
  float* part_o;              // [slots, heads_pad, D] unnormalised partial outputs
  float2* part_ml;            // [slots, heads_pad] (running max in log2 units, sum of 2^(s - max))
  unsigned int* err;          // device error word
  long long total_rows;       // T = Hkv * sum(N)
  unsigned long long cta_magic;   // ceil(2^64 / num_ctas): qda_cta_row_fast divides by num_ctas with it
  int B, H, Hkv, D, GS, NG, W, nrep, heads_pad, head_chunks, num_ctas, tile_rows, stages;
  int L;                      // query positions per sequence; head j of a KV head is (position j / nrep, j % nrep)
  int mode;                   // lean split kernel: 0 single-pass, 1 multi-query, 2 compat pass A, 3 compat pass B
  int k_only;                 // the ring carries K only (compat pass A)
  int compat;                 // merge: plain sum of the partials (compat pass B wrote normalised sums)
  int stall_chunk;            // testing aid: CTA 0's producer stops before this chunk (-1: never)
  int tile_shift;             // log2(tile_rows): pipeline tiles are powers of two
  int f16;                    // q / scales / biases are fp16 (else bf16)
  float qscale;               // log2(e) / sqrt(D): scores come out in log2 units
  int seq_off[QDA_MAX_B + 1]; // seq_off[b] = N[0] + ... + N[b-1]
};

// Query head j (0 <= j < nrep * L) of KV head kvh of sequence b: its row of q / out ([B, L, H, D] as rows of D)
// and how many of the unit's last rows it must not see (the L new tokens are causal among themselves).
__host__ __device__ inline long long qda_q_row(int b, int kvh, int j, int nrep, int L, int H) {
  const int l = j / nrep;
  return ((long long)b * L + l) * H + (long long)kvh * nrep + (j - l * nrep);
}
__host__ __device__ inline int qda_hidden_tail(int j, int nrep, int L) { return L - 1 - j / nrep; }

// Row range of CTA c: [qda_cta_row(c), qda_cta_row(c + 1)). Interior boundaries are multiples of 8 rows so that
// every scale/bias tile a CTA copies starts on a 16-byte boundary whatever the group count per row.
__host__ __device__ inline long long qda_cta_row(long long T, int C, int c) {
  if (c >= C) return T;
  if (c <= 0) return 0;
  return ((T * (long long)c) / C) & ~7LL;
}

// qda_cta_row with the division by C done as a multiply by magic = ceil(2^64 / C) (the high half of the 128-bit
// product). Exact while T * c < 2^52 and C <= 4096: the product overshoots (T * c) / C by less than
// T * c / 2^64 < 2^-12 <= 1 / C, too little to reach the next integer. T < 2^37 here (int32 sequence offsets,
// at most 64 KV heads) and C <= 4096 (the plan's cap).
__host__ __device__ inline long long qda_cta_row_fast(long long T, int C, unsigned long long magic, int c) {
  if (c >= C) return T;
  if (c <= 0) return 0;
  const unsigned long long x = (unsigned long long)T * (unsigned long long)c;
#ifdef __CUDA_ARCH__
  const unsigned long long q = __umul64hi(x, magic);
#else
  const unsigned long long q = (unsigned long long)(((unsigned __int128)x * magic) >> 64);
#endif
  return (long long)q & ~7LL;
}

// CTA whose row range holds row r (empty ranges are skipped).
__host__ __device__ inline int qda_cta_of(long long T, int C, long long r) {
  int c = (int)((r * (long long)C) / T);
  if (c >= C) c = C - 1;
  while (c + 1 < C && qda_cta_row(T, C, c + 1) <= r) ++c;
  while (c > 0 && qda_cta_row(T, C, c) > r) --c;
  return c;
}

// Shared-memory layout of the split kernel.
struct QdaSmemLayout {
  size_t codes_bytes;   // one tensor's packed codes for tile_rows rows
  size_t sc_bytes;      // one scale/bias array for tile_rows rows (multiple of 16)
  size_t stage_bytes;   // K codes, V codes, K scales, K biases, V scales, V biases
  size_t stage0;        // offset of stage 0 (after the barriers)
  size_t comb;          // offset of the cross-warp combine area
  size_t total;
};

__host__ __device__ inline QdaSmemLayout qda_smem_layout(int tile_rows, int stages, int W, int NG, int NH, int D) {
  QdaSmemLayout L;
  L.codes_bytes = (size_t)tile_rows * W * 4;
  L.sc_bytes = ((size_t)tile_rows * NG * 2 + 15) & ~(size_t)15;
  L.stage_bytes = 2 * L.codes_bytes + 4 * L.sc_bytes;
  L.stage0 = 256;
  L.comb = L.stage0 + (size_t)stages * L.stage_bytes;
  L.total = L.comb + (size_t)QDA_NW * NH * D * 4 + (size_t)QDA_NW * NH * 2 * 4;
  return L;
}

// Lean split kernel: floats of per-warp scratch (K coefficients (A, A, B, B) and V coefficients A_v, B_v per
// (row, group), p * A_v pairs per (row, head, group) with one float4 of padding per row, per-head sums of p * B_v
// per group).
// Rounded up to whole float4s: every warp's scratch starts on a 16-byte boundary (its first array is read as float4).
__host__ __device__ inline int split2_scratch_floats(int R, int NG, int NH) {
  return (R * NG * (4 + 2) + R * ((NH / 2) * NG + 1) * 4 + NH * NG + 3) & ~3;
}

// Launchers of the split kernel, translation units per (bits, exact V codes, head-dimension set): (D, heads per CTA,
// groups per row). They return cudaSuccess or the launch error.
cudaError_t qda_launch_split2_b4_x0(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_launch_split2_b4_x1(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_launch_split2_b8_x0(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_launch_split2_b8_x1(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_occupancy_split2_b4_x0(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
cudaError_t qda_occupancy_split2_b4_x1(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
cudaError_t qda_occupancy_split2_b8_x0(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
cudaError_t qda_occupancy_split2_b8_x1(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
// the D = 64 and 128 instances of the lean kernel (their own translation units)
cudaError_t qda_launch_split2s_b4_x0(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_launch_split2s_b4_x1(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_launch_split2s_b8_x0(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_launch_split2s_b8_x1(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t qda_occupancy_split2s_b4_x0(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
cudaError_t qda_occupancy_split2s_b4_x1(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
cudaError_t qda_occupancy_split2s_b8_x0(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
cudaError_t qda_occupancy_split2s_b8_x1(int D, int nh, int ng, size_t smem, int* ctas_per_sm);

// Records a CUDA runtime error for qdecode_attn_last_cuda_error() (this host thread) and returns QDA_ERR_CUDA.
int qda_cuda_fail(cudaError_t e);

// slices: CTAs per (b, l, h), each combining D / slices values of the head dimension.
cudaError_t qda_launch_merge(const QdaParams& p, void* out, int out_dtype, bool pdl, int slices, cudaStream_t s);

// Where the quantizer writes its rows. append = 0: row i to row i. append = 1 (cache append): input row
// i = ((b * Hkv) + kvh) * T + t goes to row Hkv * off_new[b] + kvh * (n_old[b] + T) + n_old[b] + t of the new cache,
// off_new[b] = sum over earlier sequences of n_old + T; off_old is the old cache's sequence starts (sum of n_old).
struct QdaRowMap {
  int append, B, Hkv, T;
  int n_old[QDA_MAX_B];
  int off_old[QDA_MAX_B + 1];
  int off_new[QDA_MAX_B + 1];
};

cudaError_t qda_launch_quantize(const float* x, long long rows, int D, int GS, int bits, int in_dtype,
                                uint32_t* packed, uint16_t* scales, uint16_t* biases, cudaStream_t s,
                                const QdaRowMap* map = nullptr);

// Copies every old row of a cache into its place in the appended cache (map->append = 1); W words and NG scales
// and biases per row, for K and V.
cudaError_t qda_launch_append_copy(const uint32_t* kp, const uint16_t* ks, const uint16_t* kb, const uint32_t* vp,
                                   const uint16_t* vs, const uint16_t* vb, uint32_t* kpo, uint16_t* kso,
                                   uint16_t* kbo, uint32_t* vpo, uint16_t* vso, uint16_t* vbo, long long rows_old,
                                   int W, int NG, const QdaRowMap& map, cudaStream_t s);
