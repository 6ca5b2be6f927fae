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
  int kstages;                // tensor-core kernel: depth of the K-code ring (stages: of the V ring)
  int L;                      // query positions per sequence; head j of a KV head is (position j / nrep, j % nrep)
  int mode;                   // lean split kernel: 0 single-pass, 1 multi-query, 2 compat pass A, 3 compat pass B
  int k_only;                 // the ring carries K only (compat pass A)
  int compat;                 // merge: plain sum of the partials (compat pass B wrote normalised sums)
  int stall_chunk;            // testing aid: CTA 0's producer stops before this chunk (-1: never)
  int tile_shift;             // log2(tile_rows): pipeline tiles are powers of two
  int f16;                    // q / scales / biases are fp16 (else bf16)
  int launch_pdl;             // host side: the lean split kernel is launched with programmatic dependent launch
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

// ---------------------------------------------------------------------- tensor-core split kernel (4-bit codes)
// Warp roles of the tensor-core split kernel (one CTA per SM): converters turn a tile's K codes into the MMA's A
// operand in tensor memory, epilogue warps turn the MMA's sums into scores and weights, V warps accumulate the V
// rows on the CUDA cores; one producer warp streams the cache, two warps issue the MMAs.
#define QDA_TC_CONV 4
#define QDA_TC_EPI 4
#define QDA_TC_VW 8
#define QDA_TC_WARPS (QDA_TC_CONV + QDA_TC_EPI + QDA_TC_VW + 3)
#define QDA_TC_THREADS (QDA_TC_WARPS * 32)
#define QDA_TC_TILE 128   // rows per pipeline tile: the M of every MMA

// Bytes of codes per ring slot of the tensor-core kernel: a slot of 32 KB of K codes (and one of V codes) holds
// 32768 / (D / 2) rows, several 128-row MMA tiles. The size is the point: bulk copies that complete a barrier phase
// per 16 KB stream the cache at about 4 TB/s on GB300, per 32 KB or more at about 7 TB/s.
#define QDA_TC_SLOT_BYTES 32768

// Rows per pipeline step of the tensor-core kernel: two 128-row MMA tiles at D = 128, one at D = 256.
__host__ __device__ inline int qda_tc_step_rows(int D) { return D == 128 ? 2 * QDA_TC_TILE : QDA_TC_TILE; }

// Rows per ring slot for head dimension D (4-bit codes: D / 2 bytes per row).
__host__ __device__ inline int qda_tc_slot_rows(int D) { return QDA_TC_SLOT_BYTES / (D / 2); }

// Shared-memory layout of the tensor-core split kernel for one (D, heads per CTA, groups per row) and ring depths:
// a ring of K-code slots (kept until converted) and a ring of V-code + scale/bias slots (kept until the scores and
// the V rows of every tile of the slot are done; a slot that ends a segment also serves as its combine area).
struct QdaTcLayout {
  size_t b_op;         // [2] B operand: q of a unit's heads, 16 x D 16-bit values in K-major core matrices
  size_t qs;           // [2][NG][NH] fp32 sums of q per group
  size_t alpha;        // [2][4][NH] fp32 rescale factors per tile, lane quarter and head
  size_t ps;           // [2][step rows][ps_row] float4: p * A_v per (row, group), four heads
  int ps_row;          // float4 per row of ps (NG, plus one against bank conflicts)
  int slot_rows;       // rows per ring slot
  size_t k_bytes;      // one K slot (slot rows x D / 2 bytes, 16-byte chunks swizzled by the tensor copy)
  size_t v_bytes;      // V codes of one slot
  size_t sc_bytes;     // one scale or bias array of a slot (slot rows x NG 16-bit values, 16-byte multiple)
  size_t vstage_bytes; // V codes, K scales, K biases, V scales, V biases
  size_t k0, v0;       // offsets of the K ring (1024-byte aligned: the swizzle follows address bits 4..9) and V ring
  size_t total;
};

// Bytes the segment-end combine needs: every V warp's o[NH][D], per lane quarter the (max, sum) per head and the
// p * B_v sums per (group, head).
__host__ __device__ inline size_t qda_tc_combine_bytes(int D, int NH, int NG) {
  return (size_t)QDA_TC_VW * NH * D * 4 + 4 * (size_t)NH * 2 * 4 + 4 * (size_t)NG * NH * 4;
}

__host__ __device__ inline QdaTcLayout qda_tc_layout(int D, int NH, int NG, int kstages, int vstages) {
  QdaTcLayout L;
  const size_t RB = (size_t)D / 2;
  L.slot_rows = qda_tc_slot_rows(D);
  L.b_op = 1024;   // barriers, the abort word and the tensor-memory address sit below
  L.qs = L.b_op + 2 * 32 * (size_t)D;
  L.alpha = L.qs + 2 * (size_t)NG * NH * 4;
  L.ps = (L.alpha + 2 * 4 * (size_t)NH * 4 + 15) & ~(size_t)15;
  L.ps_row = NG + 1;
  const size_t ps_bytes = 2 * (size_t)qda_tc_step_rows(D) * L.ps_row * 16;
  L.k_bytes = (size_t)L.slot_rows * RB;
  L.v_bytes = (size_t)L.slot_rows * RB;
  L.sc_bytes = ((size_t)L.slot_rows * NG * 2 + 15) & ~(size_t)15;
  L.vstage_bytes = L.v_bytes + 4 * L.sc_bytes;
  L.k0 = (L.ps + ps_bytes + 1023) & ~(size_t)1023;
  L.v0 = L.k0 + (size_t)kstages * L.k_bytes;
  L.total = L.v0 + (size_t)vstages * L.vstage_bytes;
  return L;
}

// Tensor-core split kernel launches (tmap_k: the CUtensorMap of the K codes, a second kernel parameter) and their
// occupancy, per output form (x1: fp32 outputs); D in {128, 256}, nh = 4, ng = D / GS >= 2.
cudaError_t qda_launch_tc_x0(const QdaParams& p, const void* tmap_k, int D, int nh, int ng, dim3 grid, size_t smem,
                             cudaStream_t s);
cudaError_t qda_launch_tc_x1(const QdaParams& p, const void* tmap_k, int D, int nh, int ng, dim3 grid, size_t smem,
                             cudaStream_t s);
cudaError_t qda_occupancy_tc_x0(int D, int nh, int ng, size_t smem, int* ctas_per_sm);
cudaError_t qda_occupancy_tc_x1(int D, int nh, int ng, size_t smem, int* ctas_per_sm);

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

// slices: CTAs per (b, l, h), each combining D / slices values of the head dimension; num_sms: the device's SMs (a
// merge of few CTAs takes 1024 threads per CTA).
cudaError_t qda_launch_merge(const QdaParams& p, void* out, int out_dtype, bool pdl, int slices, int num_sms,
                             cudaStream_t s);

// Where the quantizer writes its rows. append = 0: row i to row i. append = 1 (cache append): input row
// i = ((b * Hkv) + kvh) * T + t goes to row Hkv * off_new[b] + kvh * (n_old[b] + T) + n_old[b] + t of the new cache,
// off_new[b] = sum over earlier sequences of n_old + T; off_old is the old cache's sequence starts (sum of n_old).
struct QdaRowMap {
  int append, B, Hkv, T;
  int n_old[QDA_MAX_B];
  int off_old[QDA_MAX_B + 1];
  int off_new[QDA_MAX_B + 1];
};

// pdl: launched with programmatic dependent launch behind the previous kernel on the stream, which must not write
// anything this launch reads (the kernels of one cache append); the launch still completes after that kernel.
cudaError_t qda_launch_quantize(const float* x, long long rows, int D, int GS, int bits, int in_dtype,
                                uint32_t* packed, uint16_t* scales, uint16_t* biases, cudaStream_t s,
                                const QdaRowMap* map = nullptr, bool pdl = false);

// Copies every old row of a cache into its place in the appended cache (map->append = 1); W words and NG scales
// and biases per row, for K and V. pdl as above.
cudaError_t qda_launch_append_copy(const uint32_t* kp, const uint16_t* ks, const uint16_t* kb, const uint32_t* vp,
                                   const uint16_t* vs, const uint16_t* vb, uint32_t* kpo, uint16_t* kso,
                                   uint16_t* kbo, uint32_t* vpo, uint16_t* vso, uint16_t* vbo, long long rows_old,
                                   int W, int NG, const QdaRowMap& map, cudaStream_t s, bool pdl = false);
