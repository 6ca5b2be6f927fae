/*
 * qdecode_attn.h - single-query (L = 1) decode attention read straight from an affine-quantized KV cache,
 * on one NVIDIA GB300 (sm_103a). C ABI: plain pointers and sizes, no framework types.
 *
 * The operation (mlx-bun fused-decode-kernel.ts, header comment, fusedDecodeSdpa and MERGE_SOURCE; maya-mac
 * mlx_kernels.py, _ATTEND for the 1/sqrt(D) scale): for every sequence b and query head h, with KV head
 * kv = h / (H / Hkv),
 *
 *     out[b, h, :] = sum_n softmax_n( q[b, h, :] . k_hat[b, kv, n, :] / sqrt(D) ) * v_hat[b, kv, n, :]
 *
 * where k_hat = scale * code + bias per group of GS consecutive elements along D (maya-mac _linear_kernel 8-bit
 * load; fused-decode-kernel.ts SCORE_ROW). The dequantised cache and the score row are never written to
 * memory: the library streams the packed rows once, splits the rows of the whole batch into equal contiguous
 * ranges (one per CTA), keeps an online softmax per range and merges the ranges in a fixed order (flash-
 * decoding split-N, fused-decode-kernel.ts BLOCK_SOURCE / MERGE_SOURCE). Results are bitwise reproducible
 * from run to run for a given shape and GPU.
 *
 * Cache format (MLX affine quantization):
 *   packed  uint32 words, 32/bits codes per word, least-significant code first: element i of a row is
 *           (word[i / (32/bits)] >> (bits * (i % (32/bits)))) & (2^bits - 1).
 *   scales, biases  one per group of GS elements, stored in the input dtype (bf16 or fp16).
 *
 * Layouts (row-major, all device memory owned by the caller):
 *   q       [B, H, D]                     input dtype
 *   out     [B, H, D]                     output dtype
 *   per sequence b, back to back with no padding, starting at row Hkv * (N[0] + ... + N[b-1]):
 *     k_packed, v_packed  [Hkv, N[b], D * bits / 32]  uint32
 *     k_scales, k_biases, v_scales, v_biases  [Hkv, N[b], D / GS]  input dtype
 *   For B = 1 this is MLX's [1, Hkv, N, .] cache layout.
 *
 * Error behaviour: every function returns a status (0 = success, negative = QDA_ERR_*). Arguments are checked
 * on the host before anything is launched; a rejected call touches no GPU state. Nothing aborts, throws across
 * the ABI or traps on the device. A CUDA runtime error is returned as QDA_ERR_CUDA and kept for
 * qdecode_attn_last_cuda_error() (per host thread).
 */
#ifndef QDECODE_ATTN_H
#define QDECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QDA_OK 0
#define QDA_ERR_INVALID (-1)     /* null pointer, non-positive size, H % Hkv != 0, N[b] < 1 (N[b] < L for
                                    qdecode_attn_multi), bad dtype code */
#define QDA_ERR_UNSUPPORTED (-2) /* bits not in {4, 8}, GS not in {32, 64, 128}, D not in {64, 128, 256, 512},
                                    D % GS != 0, B > QDA_MAX_B, L * H / Hkv > QDA_MAX_NREP, L > QDA_MAX_L */
#define QDA_ERR_ALIGN (-3)       /* a data pointer is not 16-byte aligned */
#define QDA_ERR_CUDA (-4)        /* CUDA runtime error; see qdecode_attn_last_cuda_error() */
#define QDA_ERR_WORKSPACE (-5)   /* the caller-provided workspace is smaller than the call needs */
#define QDA_ERR_SCRATCH (-6)     /* qdecode_attn_noalloc: the call needs more scratch than QDA_STATIC_SCRATCH_BYTES */

#define QDA_BF16 1
#define QDA_FP16 2
#define QDA_FP32 3
/* dtype argument: input dtype (of q, scales and biases) in the low byte, output dtype in the next byte; an
   output byte of 0 means "same as the input". Input: QDA_BF16 or QDA_FP16. Output: any of the three. */
#define QDA_DTYPE(in_, out_) ((in_) | ((out_) << 8))

#define QDA_MAX_B 512
#define QDA_MAX_NREP 64
#define QDA_MAX_L 8

/*
 * qdecode_attn: decode attention for B sequences (the operation above). Asynchronous on `stream` (a
 * cudaStream_t; NULL = the legacy default stream): returns once the two kernels are enqueued and never
 * synchronises. N is a HOST array of B lengths (N[b] >= 1). The call reads q and the cache, writes out, and uses
 * a workspace of qdecode_attn_workspace_bytes() bytes: the library's own per-device buffer (allocated or grown
 * with cudaMalloc on first need, which synchronises the device) unless one was installed with
 * qdecode_attn_set_workspace(). Calls that share one workspace must not overlap on the GPU. When the library's
 * buffer grows, the smaller one is kept allocated (not freed) until the process ends, so a CUDA graph captured
 * before the growth still writes to valid memory; a captured call can also use an installed workspace or
 * qdecode_attn_noalloc, whose scratch never moves.
 *
 * Kernels: for 4-bit caches with D = 128 or 256, at least two groups per row and three or more query heads per KV
 * head, the scores of each 128-row tile are computed on the tensor cores (tcgen05: codes as exact 16-bit values
 * 128 + c (bf16) or 1024 + c (fp16), q in its own 16-bit dtype, fp32 accumulation per group); every other shape,
 * and the V side everywhere, runs on CUDA cores in fp32.
 */
int qdecode_attn(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                 const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out,
                 int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream);

/*
 * qdecode_attn_host: qdecode_attn with HOST buffers. q, the six cache arrays and out are host memory in the layouts
 * above (page-locked memory, e.g. from cudaHostAlloc, gives full-speed asynchronous copies; pageable memory works
 * and is slower). The call copies q and the cache to a device staging area, decodes with the same kernels as
 * qdecode_attn, and copies out back, all asynchronously: the result is in out once `stream` has reached the end of
 * this call's work (cudaStreamSynchronize), and the host inputs must stay unchanged until then. (The pages this
 * library follows have no counterpart of this entry point; it is the end-to-end path with the cache held on the
 * host.)
 *
 * The staging area is two sets of device buffers owned by the library (allocated or grown with cudaMalloc on first
 * need, which synchronises the device) that consecutive calls use in turn: one call's host->device copies run on a
 * library-owned copy stream and overlap the previous call's kernels on `stream`. Calls on one device are
 * serialised by a lock on the host; the call is not capturable in a CUDA graph. Returns the codes of qdecode_attn.
 */
int qdecode_attn_host(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                      const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out,
                      int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream);

/*
 * qdecode_attn_noalloc: the same operation, arguments, layouts and result as qdecode_attn, for callers that are not
 * allowed to allocate device memory at all -- for example code running under an allocator that owns the whole
 * device, a real-time loop where cudaMalloc's implicit device synchronisation is not acceptable, or a host that
 * hands this library only pre-allocated buffers. (The pages this library follows have no counterpart of this
 * entry point.)
 *
 * Its scratch space for the per-range partial results is a fixed array of QDA_STATIC_SCRATCH_BYTES compiled into
 * the library: every GPU that loads the library holds that much device memory until the process exits. No call
 * allocates or frees anything. A shape whose scratch need (qdecode_attn_workspace_bytes) exceeds the array is
 * rejected with QDA_ERR_SCRATCH before anything is launched. The first call on a device looks up the array's
 * device address and caches it (and sets the kernels' shared-memory limits): make that first call before any
 * stream capture on that device. The array is shared by every call on a device and keeps the previous call's
 * contents; nothing in it needs to start at zero, but calls whose kernels overlap on the GPU (different streams,
 * no ordering between them) race on it and must be serialised by the caller.
 */
#define QDA_STATIC_SCRATCH_BYTES (8u << 20)
int qdecode_attn_noalloc(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                         const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out,
                         int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream);

/*
 * qdecode_attn_multi: small-L multi-query decode (for example verifying L speculative tokens). Each sequence b
 * has L query positions, its last L tokens, whose K and V rows are already the last L rows of its cache (N[b]
 * counts them, so N[b] >= L). Query position l (0 <= l < L) attends the rows up to and including its own, the
 * first N[b] - L + 1 + l rows of its KV head:
 *
 *     out[b, l, h, :] = sum_{n < N[b]-L+1+l} softmax_n( q[b, l, h, :] . k_hat[b, kv, n, :] / sqrt(D) ) v_hat[b, kv, n, :]
 *
 * (The single-query kernel of mlx-bun fused-decode-kernel.ts leaves L > 1 to a separate path, header comment; the
 * matrix-vector kernels of @mlx-bun/inference trellis/reduce.ts take up to TRELLIS_MATVEC_MAX_M = 4 rows.) The L
 * positions of a KV head's query heads share one stream of its cache rows: every (position, head) pair is served
 * like one more query head of the KV head. q and out are [B, L, H, D]; everything else (cache layout, dtype,
 * workspace, stream, errors) is as for qdecode_attn, and L = 1 gives qdecode_attn's result bit for bit.
 * Requires 1 <= L <= QDA_MAX_L and L * (H / Hkv) <= QDA_MAX_NREP (else QDA_ERR_UNSUPPORTED; L < 1 or N[b] < L is
 * QDA_ERR_INVALID). Its plan and workspace size come from qdecode_attn_multi_plan.
 */
int qdecode_attn_multi(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                       const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out,
                       int B, int L, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype,
                       void* stream);

/*
 * qdecode_attn_compat: the same attention in the pages' two-pass form with their compat rounding points
 * (mlx-bun fused-decode-kernel.ts, header comment: kernel A takes per-block (max, sum-exp) over scores rounded to T,
 * kernel C sums T(exp(s - M) / denom) * dequant(V) with the full-row (M, denom), the merge sums the blocks and
 * casts to T), for comparison with MLX-style unfused paths. T is the input dtype. Per query head:
 *
 *     s_n = T(q . k_hat_n / sqrt(D))   (fp32 dot, rounded to T)
 *     p_n = T(exp(s_n - M) / denom)    (M = max_n s_n, denom = sum_n exp(s_n - M), fp32)
 *     out = sum_n p_n * v_hat_n        (fp32, not renormalised, rounded to the output dtype)
 *
 * K is read twice (once per pass), V once. Arguments, layouts, supported shapes, workspace, stream and errors as for
 * qdecode_attn.
 */
int qdecode_attn_compat(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                        const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out,
                        int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream);

/* The launch plan qdecode_attn would use (host only). Determined by the shape and the GPU alone. */
typedef struct {
  int num_ctas;           /* CTAs along the flattened row space (each takes one contiguous row range) */
  int head_chunks;        /* CTAs per row range when one CTA cannot hold all L*H/Hkv query heads of a KV head */
  int heads_per_cta;      /* query heads (position, head pairs when L > 1) a CTA serves */
  int tile_rows;          /* cache rows per pipeline stage */
  int stages;             /* pipeline depth (stages of tile_rows rows in flight per CTA) */
  int threads;            /* threads per CTA */
  int units;              /* B * Hkv (sequence, KV head) pairs */
  int smem_bytes;         /* dynamic shared memory per CTA */
  long long total_rows;   /* Hkv * (N[0] + ... + N[B-1]) */
  long long slots;        /* partial-result slots in the workspace */
  size_t workspace_bytes;
} qda_plan;

/*
 * qdecode_attn_plan: fill *plan for this shape. num_sms / ctas_per_sm describe the GPU; pass 0 for either to
 * query the current device (that needs a GPU). Same argument checks and status codes as qdecode_attn.
 */
int qdecode_attn_plan(int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int num_sms,
                      int ctas_per_sm, qda_plan* plan);

/* qdecode_attn_plan for L query positions per sequence (the plan qdecode_attn_multi uses); L = 1 is the same. */
int qdecode_attn_multi_plan(int B, int L, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int num_sms,
                            int ctas_per_sm, qda_plan* plan);

/* Workspace size in bytes that qdecode_attn and qdecode_attn_compat need for this shape on the current device,
   whatever the dtype argument (the largest over the kernels those calls can take). */
int qdecode_attn_workspace_bytes(int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, size_t* bytes);

/*
 * Install a caller-owned device workspace for the current device (16-byte aligned; ptr = NULL reverts to the
 * library's own buffer). The library never frees it. A call whose shape needs more returns QDA_ERR_WORKSPACE.
 */
int qdecode_attn_set_workspace(void* ptr, size_t bytes);

/*
 * Testing aid: force the number of row-range CTAs (0 = use the heuristic). Applies to later calls from every
 * thread. Results stay within the oracle tolerance for any split count; bitwise identity holds per split count.
 */
int qdecode_attn_debug_force_splits(int num_ctas);

/*
 * Testing aid for failure detection: with chunk >= 0, the producer of the first CTA of later calls (from every
 * thread) stops before its chunk number `chunk`, so that CTA's consumers wait for data that never comes. Their
 * bounded wait gives up after its time limit (about one second), the call's output is invalid and
 * qdecode_attn_device_status() reports bit 1; the context stays usable. chunk < 0 switches it off.
 */
int qdecode_attn_debug_stall_chunk(int chunk);

/*
 * Timing aid: when `event` (a cudaEvent_t) is non-NULL, later qdecode_attn calls from this host thread record it
 * on the stream between the split kernel and the merge kernel (the merge then launches without programmatic
 * dependent launch). NULL switches it off.
 */
int qdecode_attn_set_split_event(void* event);

/*
 * qdecode_quantize: quantize `rows` fp32 rows x [rows, D] (device) into the cache format above and write
 * packed [rows, D*bits/32] uint32, scales and biases [rows, D/GS] in the input dtype of `dtype`. Per group:
 * scale = (max - min) / (2^bits - 1) and bias = min, both computed in fp32 and stored rounded to nearest-even;
 * code = clamp(rint((x - bias) / scale), 0, 2^bits - 1) in IEEE fp32 (code 0 where the stored scale is 0).
 * Appending new tokens to a cache is this call on pointers offset to the first new row. Asynchronous on stream.
 */
int qdecode_quantize(const float* x, long long rows, int D, int GS, int bits, int dtype, uint32_t* packed,
                     void* scales, void* biases, void* stream);

/*
 * qdecode_qgemv: the cache's affine codec under a plain matrix-vector product, a comparison workload (maya-mac
 * mlx_kernels.py, _linear_kernel: weights dequantised inline as code * scale + bias per group of GS along a row):
 *
 *     y[t, n] = sum_k x[t, k] * (scale[n, k / GS] * code[n, k] + bias[n, k / GS]),   0 <= t < T
 *
 * x [T, K] and the scales and biases in the input dtype of `dtype` (bf16 or fp16); packed [N, K * bits / 32] uint32,
 * codes least-significant first; scales, biases [N, K / GS]; y [T, N] in the output dtype (as for qdecode_attn:
 * 0 = the input dtype). Asynchronous on `stream`, no workspace. Requires bits in {4, 8}, GS in {32, 64, 128},
 * 1 <= T <= QDA_QGEMV_MAX_T and K a multiple of 512 (8-bit) or 1024 (4-bit) (else QDA_ERR_UNSUPPORTED); pointers
 * 16-byte aligned.
 */
#define QDA_QGEMV_MAX_T 4
int qdecode_qgemv(const void* x, const uint32_t* w_packed, const void* w_scales, const void* w_biases, void* y,
                  int T, int N, int K, int GS, int bits, int dtype, void* stream);

/*
 * qdecode_cache_append: the cache for the next step, with T new tokens per sequence (maya-mac mlx_kernels.py,
 * _ATTEND: each pass writes the cache anew, every KV head's old rows followed by the pass's new rows). Reads the
 * cache for lengths N[b] (N[b] >= 0; with every N[b] = 0 the six old pointers may be NULL) and k_new, v_new
 * [B, Hkv, T, D] fp32 (device); writes the six *_out arrays in the same back-to-back layout for lengths N[b] + T:
 * per (b, kvh) the old rows copied unchanged, then the new rows quantized exactly as qdecode_quantize does (so the
 * result equals quantizing the longer fp32 cache). The output must not overlap the input. Same dtype argument,
 * shapes and errors as qdecode_quantize (plus B <= QDA_MAX_B); pointers 16-byte aligned. Asynchronous on stream.
 */
int qdecode_cache_append(const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                         const uint32_t* v_packed, const void* v_scales, const void* v_biases, const float* k_new,
                         const float* v_new, uint32_t* k_packed_out, void* k_scales_out, void* k_biases_out,
                         uint32_t* v_packed_out, void* v_scales_out, void* v_biases_out, int B, int Hkv,
                         const int32_t* N, int T, int D, int GS, int bits, int dtype, void* stream);

/* Human-readable text for a status code (static storage). */
const char* qdecode_attn_strerror(int status);

/* The cudaError_t behind the last QDA_ERR_CUDA returned on this host thread (0 if none). */
int qdecode_attn_last_cuda_error(void);

/*
 * Device-side status: copies (synchronously) and clears the current device's error word. Bits: 1 = a pipeline
 * wait in the split kernel gave up after its time limit (the output of that call is invalid); 2 = waiting for the
 * CTA's own copies to land before it exits gave up; 4 = an index check failed (only a library built with
 * QDA_BOUNDS_CHECK checks, and it skips the access). 0 = clean.
 */
int qdecode_attn_device_status(unsigned int* flags);

/* Number of qdecode_attn calls that launched kernels since the library was loaded (all threads). */
long long qdecode_attn_calls(void);

#ifdef __cplusplus
}
#endif

#endif /* QDECODE_ATTN_H */
