// Shared pieces of the split kernel of quantized-KV decode attention (sm_103a): the chunk walker, the producer warp
// that streams a CTA's row range through the shared-memory ring, the compat-mode helpers and the launch helpers.
//
// One CTA owns one contiguous range of the flattened cache rows (all sequences, all KV heads, back to back) and
// every query head of the KV heads in that range, so each packed byte is read from HBM exactly once. The flash-
// decoding split-N of mlx-bun fused-decode-kernel.ts (BLOCK_SOURCE: per-block running max / sum-exp /
// unnormalised o, merged later) is kept; what changes for GB300:
//   * the row space is cut into equal ranges, one per resident CTA, instead of fixed blocks per head, so a
//     ragged batch is balanced across the 152 SMs;
//   * a producer warp streams each range through a multi-stage shared-memory ring with 1-D bulk copies (TMA)
//     completing on mbarriers, the consumer warps never touch global memory for K/V;
//   * the dequantisation is factored out of the dot (SCORE_ROW: sum (s*c + b) q = s * sum c q + b * sum q) and
//     scores stay fp32, in log2 units (q is pre-scaled by log2(e)/sqrt(D)) so every exponential is one ex2.
// A range that crosses a (sequence, KV head) boundary ends one segment and starts another; each segment leaves
// one partial (max, sum, o[D]) per query head in the workspace slot (cta + unit), merged by the merge kernel.
// The consumer warps are in qda_split2.cuh.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>
#include <set>
#include <utility>

#include "qda_internal.h"
#include "qda_ptx.cuh"

namespace qda {

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A score or probability rounded to the input dtype (the compat rounding points of the two-pass form).
__device__ __forceinline__ float round_to_input(float x, bool f16) {
  return f16 ? __half2float(__float2half_rn(x)) : __bfloat162float(__float2bfloat16_rn(x));
}

// Iterates the chunks of one CTA's row range. A chunk is the intersection of one pipeline tile (tile_rows rows,
// aligned in the global row space), one (sequence, KV head) unit and the CTA's range.
struct ChunkWalker {
  long long r, r_end, u_start, u_end;
  int b, kvh, unit;

  __device__ void init(const QdaParams& p, long long r0, long long r1) {
    r = r0;
    r_end = r1;
    int lo = 0, hi = p.B - 1;  // last sequence whose first row is <= r0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)p.Hkv * p.seq_off[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const long long n = p.seq_off[b + 1] - p.seq_off[b];
    const long long sb = (long long)p.Hkv * p.seq_off[b];
    const long long off = r0 - sb;   // < Hkv * n; a 32-bit division when it fits
    kvh = off < (1LL << 31) ? (int)((unsigned)off / (unsigned)n) : (int)(off / n);
    u_start = sb + (long long)kvh * n;
    u_end = u_start + n;
    unit = b * p.Hkv + kvh;
  }

  __device__ bool next(const QdaParams& p, long long& c0, long long& c1, long long& t0) {
    if (r >= r_end) return false;
    while (r >= u_end) {
      if (++kvh == p.Hkv) { kvh = 0; ++b; }
      const long long n = p.seq_off[b + 1] - p.seq_off[b];
      u_start = u_end;
      u_end = u_start + n;
      unit = b * p.Hkv + kvh;
    }
    t0 = (r >> p.tile_shift) << p.tile_shift;
    c0 = r;
    c1 = min(min(t0 + (long long)p.tile_rows, u_end), r_end);
    r = c1;
    return true;
  }
};

// Waits for a phase with a time limit but ignores the abort flag: used to let every issued copy land before the
// CTA exits.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, unsigned int* err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 1000000000ull) { atomicOr(err, 2u); return; }
  }
}

// Fills ring slot `s` with one chunk [c0, c1) of the tile starting at row t0: the K and V codes of its rows and the
// 8-row aligned cover of its scales/biases (clipped to the arrays' end; a ragged last < 16 bytes go by plain loads,
// published by the arrive), all completing on full[s]. Lane 0 posts the byte count; lanes 0..5 then issue the six
// copies side by side. Called by all 32 lanes of one warp.
__device__ __forceinline__ void issue_chunk(const QdaParams& p, unsigned char* smem, const QdaSmemLayout& L,
                                            uint64_t* full, int s, long long c0, long long c1, long long t0,
                                            long long T, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  const int NG = p.NG, W = p.W;
  const uint32_t RB = W * 4, SB = NG * 2;
  unsigned char* st = smem + L.stage0 + (size_t)s * L.stage_bytes;
  const uint32_t cbytes = (uint32_t)(c1 - c0) * RB;
  const size_t coff = (size_t)(c0 - t0) * RB;
  const long long s0 = c0 & ~7LL;
  const long long s1 = min((c1 + 7) & ~7LL, T);
  const uint32_t sbytes = (uint32_t)(s1 - s0) * SB;
  const uint32_t s16 = sbytes & ~15u;
  const size_t soff = (size_t)(s0 - t0) * SB;
  const int arrays = p.k_only ? 2 : 4;   // scale/bias arrays copied: K's, and V's unless the ring carries K only
  // the chunk lies in the tile and the arrays; else (checked build) the phase completes with no bytes
  const bool inb = in_bounds(c0 >= t0 && c0 < c1 && c1 <= T && s1 <= T && coff + cbytes <= L.codes_bytes &&
                             s0 >= t0 && soff + sbytes <= L.sc_bytes, p.err);
  if (lane == 0 && !inb) mbar_arrive_expect_tx(&full[s], 0);
  if (!inb) return;
  if (lane == 0) {
    if (s16 != sbytes) {
      const uint16_t* srcs[4] = {p.ks, p.kb, p.vs, p.vb};
      for (int a = 0; a < arrays; ++a) {
        const uint16_t* src = srcs[a] + s0 * NG + s16 / 2;
        uint16_t* dst = reinterpret_cast<uint16_t*>(st + 2 * L.codes_bytes + a * L.sc_bytes + soff + s16);
        for (uint32_t k = 0; k < (sbytes - s16) / 2; ++k) dst[k] = src[k];
      }
    }
    mbar_arrive_expect_tx(&full[s], (p.k_only ? 1 : 2) * cbytes + arrays * s16);
  }
  __syncwarp();
  if (lane == 0) {
    bulk_g2s(st + coff, p.kp + c0 * W, cbytes, &full[s], pol);
  } else if (lane == 1) {
    if (!p.k_only) bulk_g2s(st + L.codes_bytes + coff, p.vp + c0 * W, cbytes, &full[s], pol);
  } else if (lane < 2 + arrays && s16) {
    const int a = lane - 2;
    const uint16_t* src = a == 0 ? p.ks : a == 1 ? p.kb : a == 2 ? p.vs : p.vb;
    bulk_g2s(st + 2 * L.codes_bytes + a * L.sc_bytes + soff, src + s0 * NG, s16, &full[s], pol);
  }
}

// The producer warp: walks the CTA's chunks and fills the shared-memory ring. Lane 0 waits for the consumers to
// free a stage (empty[stage]) before the chunk is issued into it. Before returning, lane 0 waits until every copy
// the warp issued has landed. Called by all 32 lanes of the warp.
__device__ __forceinline__ void produce_range(const QdaParams& p, ChunkWalker walk, unsigned char* smem,
                                              const QdaSmemLayout& L, uint64_t* full, uint64_t* empty,
                                              volatile int* abort_flag, long long T) {
  const int lane = threadIdx.x & 31;
  const int STAGES = p.stages;
  const uint64_t pol = policy_evict_first();
  long long c0, c1, t0;
  int i = 0;
  int s = 0, ph = 0;   // ring slot of chunk i and the parity of its use (i / STAGES) & 1
  while (walk.next(p, c0, c1, t0)) {
    if (blockIdx.x == 0 && i == p.stall_chunk) break;   // testing aid: the consumers' wait for it must run out
    if (i == 1) {
      // the second chunk goes out once the first has landed: every CTA's first chunk then comes in one short burst
      // ahead of the rest, so the consumers start sooner (the ring still fills while they work on it)
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&full[0], 0, abort_flag, p.err, 1u);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
    if (i >= STAGES) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, p.err, 1u);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
    issue_chunk(p, smem, L, full, s, c0, c1, t0, T, pol);
    ++i;
    if (++s == STAGES) {
      s = 0;
      ph ^= 1;
    }
  }
  if (lane == 0)
    for (int j = (i > STAGES ? i - STAGES : 0); j < i; ++j) mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1, p.err);
}

// Launches kern, with programmatic dependent launch behind the previous kernel on the stream when pdl is set (the
// kernel waits, griddepcontrol.wait, before its first global-memory access; without the attribute that wait returns
// at once).
template <typename K, typename... Args>
cudaError_t launch_pdl(K kern, dim3 grid, unsigned threads, size_t smem, cudaStream_t s, bool pdl, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Raises a kernel's dynamic shared-memory limit to the opt-in maximum, once per (kernel, device).
template <typename K>
cudaError_t ensure_smem_limit(K kern, size_t smem) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  (void)smem;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_pair(reinterpret_cast<const void*>(kern), dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  done.insert(key);
  return cudaSuccess;
}

}  // namespace qda
