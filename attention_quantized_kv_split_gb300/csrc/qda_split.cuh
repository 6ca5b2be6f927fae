// Split kernel of quantized-KV decode attention (sm_103a).
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

// The (max, sum) of one head's scores over a whole unit, from pass A's per-range partials (compat pass B): the 32
// lanes take the unit's slots in turn and fold across the warp in a fixed order. Every lane gets the result.
__device__ __forceinline__ void unit_stats(const QdaParams& p, long long T, long long u_start, long long u_end,
                                           int unit, int head, float& M, float& den) {
  const int C = p.num_ctas;
  const int cf = qda_cta_of(T, C, u_start);
  const int ns = qda_cta_of(T, C, u_end - 1) - cf + 1;
  const bool maybe_empty = T / C < 8;   // only ranges shorter than 8 rows can be empty (and wrote no slot)
  M = -INFINITY;
  den = 0.f;
  for (int k = threadIdx.x & 31; k < ns; k += 32) {
    const int c = cf + k;
    if (maybe_empty && qda_cta_row(T, C, c) == qda_cta_row(T, C, c + 1)) continue;
    if (!in_bounds(c + unit < C + p.B * p.Hkv && head < p.heads_pad, p.err)) continue;
    const float2 ml = p.part_ml[(size_t)(c + unit) * p.heads_pad + head];
    const float mn = fmaxf(M, ml.x);
    den = (M == -INFINITY ? 0.f : den * exp2f(M - mn)) + ml.y * exp2f(ml.x - mn);
    M = mn;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float Mo = __shfl_xor_sync(0xffffffffu, M, off);
    const float Do = __shfl_xor_sync(0xffffffffu, den, off);
    const float mn = fmaxf(M, Mo);
    den = (M == -INFINITY ? 0.f : den * exp2f(M - mn)) + (Mo == -INFINITY ? 0.f : Do * exp2f(Mo - mn));
    M = mn;
  }
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

// BITS: 4 or 8. WPL: packed words per lane per row. LPR: lanes per row (RPS = 32/LPR rows per warp step).
// NH: query heads per CTA. D = LPR * WPL * 32 / BITS. MODE: 0 single-pass (any L), 2 compat pass A (K only,
// per-range (max, sum) of the scores rounded to the input dtype), 3 compat pass B (rounded exp(s - M) / denom times
// V, summed without rescaling).
template <int BITS, int WPL, int LPR, int NH, int MODE = 0>
__global__ void __launch_bounds__(QDA_THREADS) qda_split_kernel(const __grid_constant__ QdaParams p) {
  constexpr bool STATS = MODE == 2, APPLY = MODE == 3, COMPAT = MODE >= 2;
  constexpr float LOG2E = 1.4426950408889634f;
  constexpr int PER = 32 / BITS;          // codes per word
  constexpr int E = WPL * PER;            // elements per lane per row
  constexpr int RPS = 32 / LPR;           // rows per warp step
  constexpr int W = LPR * WPL;            // words per row
  constexpr int D = W * PER;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  constexpr int NW = QDA_NW;

  extern __shared__ __align__(1024) unsigned char smem[];
  const int TILE = p.tile_rows, STAGES = p.stages, NG = p.NG;
  const QdaSmemLayout L = qda_smem_layout(TILE, STAGES, W, NG, NH, D);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);
  float* comb_o = reinterpret_cast<float*>(smem + L.comb);
  float* comb_m = comb_o + NW * NH * D;
  float* comb_l = comb_m + NW * NH;

  const bool f16 = p.f16 != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // head chunks of one row range are adjacent blocks, so a second chunk re-reads rows while they are in L2
  const int cta = blockIdx.x / p.head_chunks, hc = blockIdx.x - cta * p.head_chunks;
  const long long T = p.total_rows;
  const long long r0 = qda_cta_row_fast(T, p.num_ctas, p.cta_magic, cta);
  const long long r1 = qda_cta_row_fast(T, p.num_ctas, p.cta_magic, cta + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (r0 >= r1) return;

  ChunkWalker walk;
  walk.init(p, r0, r1);
  long long c0, c1, t0;

  if (warp == NW) {
    produce_range(p, walk, smem, L, full, empty, abort_flag, T);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int rir = lane / LPR;     // row of the warp step this lane works on
  const int lir = lane % LPR;     // lane's slice of the row: elements [lir*E, lir*E + E)
  float qv[NH][E], qsum[NH], o[NH][E], m[NH], l[NH];
  int hide[NH];   // last rows of the unit each head must not see (multi-query decode)
  float inv[NH];  // APPLY: 1 / the unit's sum of 2^(s - m) per head
  int cur_unit = -1;
  int s = 0, phase = 0;   // ring slot of the current chunk and the parity of its use
  while (walk.next(p, c0, c1, t0)) {
    if (walk.unit != cur_unit) {  // a new (sequence, KV head): load its query heads, reset the softmax state
      cur_unit = walk.unit;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int j = hc * NH + h;
        float acc = 0.f;
        hide[h] = qda_hidden_tail(j, p.nrep, p.L);
        if (j < p.nrep * p.L &&
            in_bounds(qda_q_row(walk.b, walk.kvh, j, p.nrep, p.L, p.H) < (long long)p.B * p.L * p.H, p.err)) {
          const uint16_t* qp = reinterpret_cast<const uint16_t*>(p.q) +
                               qda_q_row(walk.b, walk.kvh, j, p.nrep, p.L, p.H) * D + lir * E;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            qv[h][e] = half_bits_to_float_rt(qp[e], f16) * p.qscale;
            acc += qv[h][e];
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) qv[h][e] = 0.f;
        }
        qsum[h] = acc;
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[h][e] = 0.f;
        if constexpr (APPLY) {   // pass B: the unit's statistics from pass A fix every weight in advance
          float den;
          unit_stats(p, T, walk.u_start, walk.u_end, walk.unit, hc * NH + h, m[h], den);
          inv[h] = 1.f / den;
        }
      }
    }
    const bool ok = mbar_wait_bounded(&full[s], phase, abort_flag, p.err, 1u);
    if (ok) {
      const unsigned char* st = smem + L.stage0 + (size_t)s * L.stage_bytes;
      const uint32_t* sK = reinterpret_cast<const uint32_t*>(st);
      const uint32_t* sV = reinterpret_cast<const uint32_t*>(st + L.codes_bytes);
      const uint16_t* sKS = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes);
      const uint16_t* sKB = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes + L.sc_bytes);
      const uint16_t* sVS = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes + 2 * L.sc_bytes);
      const uint16_t* sVB = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes + 3 * L.sc_bytes);
      const int g = (lir * E) / p.GS;
      for (long long rb = c0 + warp * RPS; rb < c1; rb += NW * RPS) {
        const long long row = rb + rir;
        const bool valid = row < c1;
        const int lr = (int)((valid ? row : c0) - t0);
        if (!in_bounds(lr >= 0 && lr < TILE, p.err)) continue;
        // K: factored dot over this lane's slice, then the sum over the LPR lanes of the row
        float cf[E];
#pragma unroll
        for (int w = 0; w < WPL; ++w) {
          const uint32_t word = sK[lr * W + lir * WPL + w];
#pragma unroll
          for (int k = 0; k < PER; ++k)
            cf[w * PER + k] = __uint_as_float(0x4B000000u | ((word >> (BITS * k)) & MASK)) - 8388608.0f;
        }
        const float ksc = half_bits_to_float_rt(sKS[lr * NG + g], f16);
        const float kbi = half_bits_to_float_rt(sKB[lr * NG + g], f16);
        float sc[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) acc = fmaf(cf[e], qv[h][e], acc);
          sc[h] = fmaf(ksc, acc, kbi * qsum[h]);
        }
#pragma unroll
        for (int h = 0; h < NH; ++h) {
#pragma unroll
          for (int off = LPR / 2; off >= 1; off >>= 1) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], off);
        }
        // online softmax over the rows of this step (one running max per head, shared by the warp)
        float pr[NH], alpha[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const bool seen = valid && row < walk.u_end - hide[h];
          float sv = sc[h];
          if constexpr (COMPAT) sv = round_to_input(sv, f16) * LOG2E;   // natural units, rounded, then log2 units
          const float sh = seen ? sv : -INFINITY;
          if constexpr (APPLY) {
            alpha[h] = 1.f;
            pr[h] = seen ? round_to_input(ex2(sh - m[h]) * inv[h], f16) : 0.f;
            continue;
          }
          float mx = sh;
#pragma unroll
          for (int off = LPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          const float mn = fmaxf(m[h], mx);
          if (mn == -INFINITY) {
            alpha[h] = 1.f;
            pr[h] = 0.f;
          } else {
            alpha[h] = ex2(m[h] - mn);
            pr[h] = seen ? ex2(sh - mn) : 0.f;
          }
          m[h] = mn;
          l[h] = fmaf(l[h], alpha[h], pr[h]);
        }
        // V: o = alpha * o + p * (s * c + b) (none in compat pass A)
        if constexpr (!STATS) {
#pragma unroll
          for (int w = 0; w < WPL; ++w) {
            const uint32_t word = sV[lr * W + lir * WPL + w];
#pragma unroll
            for (int k = 0; k < PER; ++k)
              cf[w * PER + k] = __uint_as_float(0x4B000000u | ((word >> (BITS * k)) & MASK)) - 8388608.0f;
          }
          const float vsc = half_bits_to_float_rt(sVS[lr * NG + g], f16);
          const float vbi = half_bits_to_float_rt(sVB[lr * NG + g], f16);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float ps = pr[h] * vsc, pb = pr[h] * vbi;
#pragma unroll
            for (int e = 0; e < E; ++e) o[h][e] = fmaf(o[h][e], alpha[h], fmaf(ps, cf[e], pb));
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    if (c1 == walk.u_end || c1 == r1) {
      // ------------------------------------------------------------ end of a segment: combine the warps
      if constexpr (RPS > 1) {
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
            if constexpr (!STATS) {
#pragma unroll
              for (int e = 0; e < E; ++e) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], off);
            }
          }
        }
      }
      if (!STATS && rir == 0) {
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
          for (int e = 0; e < E; ++e) comb_o[(warp * NH + h) * D + lir * E + e] = o[h][e];
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          comb_m[warp * NH + h] = m[h];
          comb_l[warp * NH + h] = l[h];
        }
      }
      named_barrier_sync(1, NW * 32);
      const long long slot = (long long)cta + walk.unit;
      // compat pass A writes only (max, sum) per head; pass B only o (other CTAs of pass B may still be reading
      // pass A's statistics)
      for (int idx = threadIdx.x; idx < (STATS ? NH : NH * D); idx += NW * 32) {
        const int h = STATS ? idx : idx / D, d = STATS ? 0 : idx - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, comb_m[w * NH + h]);
        float O = 0.f, Ls = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float mw = comb_m[w * NH + h];
          const float wt = APPLY ? 1.f : (mw == -INFINITY) ? 0.f : ex2(mw - M);
          if constexpr (!STATS) O = fmaf(comb_o[(w * NH + h) * D + d], wt, O);
          Ls = fmaf(comb_l[w * NH + h], wt, Ls);
        }
        const size_t hp = (size_t)slot * p.heads_pad + (size_t)hc * NH + h;
        if (!in_bounds(slot < (long long)p.num_ctas + p.B * p.Hkv && hc * NH + h < p.heads_pad, p.err)) continue;
        if constexpr (!STATS) p.part_o[hp * D + d] = O;
        if (!APPLY && d == 0) p.part_ml[hp] = make_float2(M, Ls);
      }
      named_barrier_sync(1, NW * 32);
    }
    if (++s == STAGES) {
      s = 0;
      phase ^= 1;
    }
  }
}

// Calls f(kernel) with the instantiation for (wpl, lpr, nh); returns cudaErrorInvalidValue for an unbuilt one.
template <int BITS, int MODE, typename Fn>
cudaError_t with_split_kernel_m(int wpl, int lpr, int nh, Fn&& f) {
#define QDA_NH_CASES(WPL_, LPR_)                                                        \
  switch (nh) {                                                                         \
    case 1: return f(qda_split_kernel<BITS, WPL_, LPR_, 1, MODE>);                 \
    case 2: return f(qda_split_kernel<BITS, WPL_, LPR_, 2, MODE>);                 \
    case 4: return f(qda_split_kernel<BITS, WPL_, LPR_, 4, MODE>);                 \
    case 8:                                                                             \
      if constexpr (WPL_ * (32 / BITS) * 8 <= 64) return f(qda_split_kernel<BITS, WPL_, LPR_, 8, MODE>); \
      else return cudaErrorInvalidValue;                                                \
    default: return cudaErrorInvalidValue;                                              \
  }
  if constexpr (BITS == 4) {
    if (wpl == 1 && lpr == 8) { QDA_NH_CASES(1, 8) }
    if (wpl == 1 && lpr == 16) { QDA_NH_CASES(1, 16) }
    if (wpl == 1 && lpr == 32) { QDA_NH_CASES(1, 32) }
    if (wpl == 2 && lpr == 32) { QDA_NH_CASES(2, 32) }
  } else {
    if (wpl == 1 && lpr == 16) { QDA_NH_CASES(1, 16) }
    if (wpl == 1 && lpr == 32) { QDA_NH_CASES(1, 32) }
    if (wpl == 2 && lpr == 32) { QDA_NH_CASES(2, 32) }
    if (wpl == 4 && lpr == 32) { QDA_NH_CASES(4, 32) }
  }
#undef QDA_NH_CASES
  return cudaErrorInvalidValue;
}

// The general kernel serves D in {64, 128} (and any shape the lean kernel does not take); mode 1 (multi-query)
// runs as mode 0, which masks at run time.
template <int BITS, typename Fn>
cudaError_t with_split_kernel(int wpl, int lpr, int nh, int mode, Fn&& f) {
  switch (mode) {
    case 0: case 1: return with_split_kernel_m<BITS, 0>(wpl, lpr, nh, f);
    case 2: return with_split_kernel_m<BITS, 2>(wpl, lpr, nh, f);
    case 3: return with_split_kernel_m<BITS, 3>(wpl, lpr, nh, f);
    default: return cudaErrorInvalidValue;
  }
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

template <int BITS>
cudaError_t launch_split(const QdaParams& p, int wpl, int lpr, int nh, dim3 grid, size_t smem, cudaStream_t s) {
  return with_split_kernel<BITS>(wpl, lpr, nh, p.mode, [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_limit(kern, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, QDA_THREADS, smem, s>>>(p);
    return cudaGetLastError();
  });
}

template <int BITS>
cudaError_t occupancy_split(int wpl, int lpr, int nh, size_t smem, int* n) {
  return with_split_kernel<BITS>(wpl, lpr, nh, 0, [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_limit(kern, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, QDA_THREADS, smem);
  });
}

}  // namespace qda
