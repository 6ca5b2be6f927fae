// Split kernel, arithmetic-lean variant: D = 64, 128 and 256 with 2 or 4 query heads per CTA, D = 512 with 2
// (sm_103a).
//
// One contiguous row range per CTA, a producer warp streaming it with bulk copies into a shared-memory ring
// (qda_split.cuh), one partial per (segment, query head); the consumer warps are organised around the instruction
// count per cache row, which bounds this path once the bytes stream at HBM speed:
//   * codes become floats with one byte permute each: 4-bit codes as 0.5 + c/256 (K, and V for 16-bit outputs),
//     8-bit codes as 1 + c/32768 (K for 16-bit outputs), or exactly as c (2^23 + c minus 2^23) where an fp32
//     output needs it; the constant offset is folded into per-row coefficients A, B with
//     s*c + b = A*f + B, computed once per (row, group) by the warp before its rows are used;
//   * every dot product and every V update is a packed two-lane FMA (f32x2);
//   * K rows are read by D/16 lanes (16 codes each) and the per-row sums are formed by a transposed butterfly,
//     so each lane ends with whole scores for fixed (rows, head) instead of every lane reducing every score;
//   * V rows are read by 32 lanes (D/32 codes each), or at D = 128 and 64 by 16 and 8 lanes of 8 codes, which then
//     take 2 and 4 rows a step and add their sums at the segment end;
//   * the online softmax advances once per block of R rows per warp (one max, one rescale of o when it moves);
//   * the lane that owns a score also forms p * A_v for every group of that row (the V coefficient of the
//     mlx-bun SCORE_ROW factoring, applied to V) and keeps the sum of p * B_v, so the V lanes only load them.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "qda_split.cuh"

namespace qda {

// ----------------------------------------------------------------------------- code -> float conversions

// 4-bit, one word (8 codes, code k at bits 4k..4k+3) -> 4 pairs (code 2j, code 2j+1).
template <bool EXACT>
__device__ __forceinline__ void unpack4(uint32_t w, float2 (&f)[4]) {
  const uint32_t lo = w & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6 in bytes 0..3
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
  if constexpr (EXACT) {
    // bytes [code, 0, 0, 0x4B] = 2^23 + code
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t sel = 0x7650u | (uint32_t)j;
      f[j] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, sel)),
                                    __uint_as_float(__byte_perm(hi, 0x4B000000u, sel))),
                        make_float2(-8388608.0f, -8388608.0f));
    }
  } else {
    // bytes [0, 0, code, 0x3F] = 0.5 + code / 256
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t sel = 0x7054u | ((uint32_t)j << 8);
      f[j] = make_float2(__uint_as_float(__byte_perm(lo, 0x3F000000u, sel)),
                         __uint_as_float(__byte_perm(hi, 0x3F000000u, sel)));
    }
  }
}

// 8-bit, one word (4 codes, code k in byte k) -> 2 pairs.
template <bool EXACT>
__device__ __forceinline__ void unpack8(uint32_t w, float2 (&f)[2]) {
  if constexpr (EXACT) {
    f[0] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u)),
                                  __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7651u))),
                      make_float2(-8388608.0f, -8388608.0f));
    f[1] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7652u)),
                                  __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7653u))),
                      make_float2(-8388608.0f, -8388608.0f));
  } else {
    // bytes [0, code, 0x80, 0x3F] = 1 + code / 32768
    f[0] = make_float2(__uint_as_float(__byte_perm(w, 0x3F800000u, 0x7604u)),
                       __uint_as_float(__byte_perm(w, 0x3F800000u, 0x7614u)));
    f[1] = make_float2(__uint_as_float(__byte_perm(w, 0x3F800000u, 0x7624u)),
                       __uint_as_float(__byte_perm(w, 0x3F800000u, 0x7634u)));
  }
}

// A word array -> NW2 * (32/BITS) / 2 pairs.
template <int BITS, bool EXACT, int NWORDS>
__device__ __forceinline__ void unpack_words(const uint32_t (&w)[NWORDS], float2 (&f)[NWORDS * 16 / BITS]) {
#pragma unroll
  for (int k = 0; k < NWORDS; ++k) {
    if constexpr (BITS == 4) {
      float2 t[4];
      unpack4<EXACT>(w[k], t);
#pragma unroll
      for (int j = 0; j < 4; ++j) f[4 * k + j] = t[j];
    } else {
      float2 t[2];
      unpack8<EXACT>(w[k], t);
#pragma unroll
      for (int j = 0; j < 2; ++j) f[2 * k + j] = t[j];
    }
  }
}

// s * c + b = A * f + B for the encoding above.
template <int BITS, bool EXACT>
__device__ __forceinline__ float2 coeffs(float s, float b) {
  if constexpr (EXACT) {
    return make_float2(s, b);
  } else if constexpr (BITS == 4) {
    return make_float2(256.0f * s, fmaf(-128.0f, s, b));
  } else {
    return make_float2(32768.0f * s, fmaf(-32768.0f, s, b));
  }
}

// The same for two groups at once: (s, b) pairs -> A in .x, B in .y of the
// results' pairs (A pair, B pair).
template <int BITS, bool EXACT>
__device__ __forceinline__ void coeffs2(float2 s, float2 b, float2& A, float2& B) {
  if constexpr (EXACT) {
    A = s;
    B = b;
  } else if constexpr (BITS == 4) {
    A = __fmul2_rn(make_float2(256.0f, 256.0f), s);
    B = __ffma2_rn(make_float2(-128.0f, -128.0f), s, b);
  } else {
    A = __fmul2_rn(make_float2(32768.0f, 32768.0f), s);
    B = __ffma2_rn(make_float2(-32768.0f, -32768.0f), s, b);
  }
}

template <int N>
__device__ __forceinline__ void load_words(const uint32_t* src, uint32_t (&w)[N]) {
  if constexpr (N == 1) {
    w[0] = src[0];
  } else if constexpr (N == 2) {
    const uint2 t = *reinterpret_cast<const uint2*>(src);
    w[0] = t.x;
    w[1] = t.y;
  } else {
#pragma unroll
    for (int k = 0; k < N; k += 4) {
      const uint4 t = *reinterpret_cast<const uint4*>(src + k);
      w[k] = t.x;
      w[k + 1] = t.y;
      w[k + 2] = t.z;
      w[k + 3] = t.w;
    }
  }
}

// Geometry of the lean variant, shared by the kernel and the host.
template <int BITS, int D, int NH>
struct Split2Geom {
  static constexpr int EK = 16;                 // K codes per lane per row
  static constexpr int LK = D / EK;             // lanes per K row (4, 8, 16 or 32)
  static constexpr int RPS = 32 / LK;           // K rows per warp step
  static constexpr int R = NH == 4 ? 8 : 16;  // rows per warp block (fewer live scores with 4 heads)
  static constexpr int S = R / RPS;             // K steps per block
  static constexpr int NV = NH * S;             // partial scores per lane before the reduction
  static constexpr int NVL = NV / LK;           // scores per lane after it
  static constexpr int EV = D >= 256 ? D / 32 : 8;   // V codes per lane per row (at least one word of 4-bit codes)
  static constexpr int VL = D / EV;             // lanes per V row (32, or 16 / 8 at D = 128 / 64)
  static constexpr int VR = 32 / VL;            // V rows per warp step
  static constexpr int KW = EK * BITS / 32;     // K words per lane per row
  static constexpr int VW = EV * BITS / 32;     // V words per lane per row
  static constexpr int W = D * BITS / 32;       // words per row
  static constexpr int TILE = QDA_SPLIT2_TILE;  // rows per pipeline stage (TILE / R blocks, dealt to the warps)
  static_assert(TILE % (R * QDA_NW) == 0, "every warp takes the same number of blocks of a full chunk");
  static_assert(NVL >= 1, "reduction must end with at least one score per lane");
  static_assert(R % VR == 0, "the V steps cover the block's rows");
};

// MODE 0: single-pass decode. 1: single-pass with L > 1 query positions (the last L - 1 rows of a unit hidden
// from some heads). 2: compat pass A, K only: per segment and head the (reference max, sum) of the scores rounded to
// the input dtype. 3: compat pass B: probabilities exp(s - M) / denom from pass A's statistics, rounded to the input
// dtype, times V, summed without rescaling (mlx-bun fused-decode-kernel.ts header: kernels A and C of the
// two-pass form).
template <int BITS, int D, int NH, int NG, bool EXACT, int MODE>
__global__ void __launch_bounds__(QDA_THREADS, 2) qda_split2_kernel(const __grid_constant__ QdaParams p) {
  using G = Split2Geom<BITS, D, NH>;
  constexpr int EK = G::EK, LK = G::LK, RPS = G::RPS, R = G::R, S = G::S, NV = G::NV, NVL = G::NVL;
  constexpr int EV = G::EV, KW = G::KW, VW = G::VW, W = G::W, VL = G::VL, VR = G::VR;
  constexpr int NW = QDA_NW;
  constexpr int LOG_NH = NH == 4 ? 2 : 1;
  constexpr int LOG_LK = LK == 32 ? 5 : LK == 16 ? 4 : LK == 8 ? 3 : 2;
  constexpr bool MULTI = MODE == 1, STATS = MODE == 2, APPLY = MODE == 3, COMPAT = MODE >= 2;
  // exact K codes where scores must be accurate to fp32: fp32 outputs with 8-bit codes (4-bit K scores are
  // accurate enough in the cheap form), and the compat passes, which round every score to the input dtype and must
  // take the same rounding decisions as a plain fp32 dot
  constexpr bool EXACT_K = (EXACT && BITS == 8) || COMPAT;
  constexpr float LOG2E = 1.4426950408889634f;

  extern __shared__ __align__(1024) unsigned char smem[];
  // the host plans this kernel with a 64-row tile; the 4-head and D = 512 kernels take it as a constant (every
  // stage and block offset folds, which frees registers), the 2-head D = 256 ones from the parameters (measured
  // faster there)
  const int TILE = (NH == 4 || D == 512) ? G::TILE : p.tile_rows;
  const int STAGES = p.stages;
  const bool f16 = p.f16 != 0;
  const QdaSmemLayout L = qda_smem_layout(TILE, STAGES, W, NG, NH, D);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);
  float* scratch_all = reinterpret_cast<float*>(smem + L.comb);   // per-warp scratch, reused as combine area
  float* comb_o = scratch_all;
  float* comb_m = comb_o + NW * NH * D;
  float* comb_l = comb_m + NW * NH;

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
  // everything above is CTA-local; when launched with programmatic dependent launch (the compat form's second pass),
  // the grid before this one on the stream is complete and visible from here on (otherwise the wait returns at once)
  pdl_wait();
  pdl_launch_dependents();
  if (r0 >= r1) return;

  ChunkWalker walk;
  walk.init(p, r0, r1);
  long long c0, c1, t0;

  if (warp == NW) {
    produce_range(p, walk, smem, L, full, empty, abort_flag, T);
    return;
  }

  // ------------------------------------------------------------------------------ consumer warp state
  const int sw_floats = split2_scratch_floats(R, NG, NH);
  float* sAB = scratch_all + warp * sw_floats;          // [R][NG] float4 (A, A, B, B) of K
  float* sAV = sAB + R * NG * 4;                        // [R][NG] A_v
  float* sBV = sAV + R * NG;                            // [R][NG] B_v
  // p * A_v as float4 (pA_h, pA_h, pA_h+1, pA_h+1) per (row, head pair, group), rows padded by one float4 so
  // that the owners of different rows write to different banks
  float* sPS = sBV + R * NG;
  constexpr int PS_ROW = (NH / 2) * NG + 1;             // float4 per row
  float* sPB = sPS + R * PS_ROW * 4;                    // [NH][NG]

  const int klane = lane & (LK - 1);                    // K slice: codes [klane*EK, klane*EK + EK)
  const int khalf = lane / LK;                          // which row of a K step
  const int gk = (klane * EK) / p.GS;
  // V slice: codes [vlane*EV, vlane*EV + EV) of the rows vrow, vrow + VR, ... of a block (VR = 1 at D >= 256)
  const int vlane = lane % VL, vrow = lane / VL;
  const int gv = (vlane * EV) / p.GS;

  // the head and rows this lane owns after the reduction
  int my_h = 0;
#pragma unroll
  for (int k = 0; k < LOG_NH; ++k) my_h += ((lane >> k) & 1) * (NH >> (k + 1));
  int my_s[NVL];
#pragma unroll
  for (int i = 0; i < NVL; ++i) {
    int s = i;
#pragma unroll
    for (int k = LOG_NH; k < LOG_LK; ++k) s += ((lane >> k) & 1) * (NV >> (k + 1));
    my_s[i] = s;  // index within the head's S steps (index - h * S)
  }
  int head_lane[NH];   // a lane that owns head h
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    int l = 0;
#pragma unroll
    for (int k = 0; k < LOG_NH; ++k) l |= ((h >> (LOG_NH - 1 - k)) & 1) << k;
    head_lane[h] = l;
  }

  float2 qk[NH][EK / 2];    // q slice for K, pre-scaled to log2 units
  float qs[NH];             // its sum (bias term)
  float2 o[NH][EV / 2];     // V accumulators
  float m_run = -INFINITY;  // running max of my head (equal across the lanes owning it)
  int my_hide = 0;          // last rows of the unit my head must not see (MULTI)
  float l_run = 0.f;        // sum of 2^(s - m_run) over my rows
  float inv_den = 0.f;      // APPLY: 1 / sum of 2^(s - m_run) over the whole unit, m_run its pass-A reference
  float pb[NG];             // sum of p * B_v per group, my head
  int cur_unit = -1;
  int stage = 0, phase = 0;   // ring slot of the current chunk and the parity of its use

  while (walk.next(p, c0, c1, t0)) {
    if (walk.unit != cur_unit) {
      cur_unit = walk.unit;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int j = hc * NH + h;
        float acc = 0.f;
        if (j < p.nrep * p.L &&
            in_bounds(qda_q_row(walk.b, walk.kvh, j, p.nrep, p.L, p.H) < (long long)p.B * p.L * p.H, p.err)) {
          const uint16_t* qp = reinterpret_cast<const uint16_t*>(p.q) +
                               qda_q_row(walk.b, walk.kvh, j, p.nrep, p.L, p.H) * D + klane * EK;
          const uint4 a = reinterpret_cast<const uint4*>(qp)[0];
          const uint4 b = reinterpret_cast<const uint4*>(qp)[1];
          const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float x = half_bits_to_float_rt(u[k] & 0xFFFFu, f16) * p.qscale;
            const float y = half_bits_to_float_rt(u[k] >> 16, f16) * p.qscale;
            qk[h][k] = make_float2(x, y);
            acc += x + y;
          }
        } else {
#pragma unroll
          for (int k = 0; k < EK / 2; ++k) qk[h][k] = make_float2(0.f, 0.f);
        }
        qs[h] = acc;
#pragma unroll
        for (int k = 0; k < EV / 2; ++k) o[h][k] = make_float2(0.f, 0.f);
      }
      m_run = -INFINITY;
      l_run = 0.f;
      if constexpr (MULTI) my_hide = qda_hidden_tail(hc * NH + my_h, p.nrep, p.L);
#pragma unroll
      for (int g = 0; g < NG; ++g) pb[g] = 0.f;
      if constexpr (APPLY) {
        // the unit's (max, sum) from pass A's partials of every range that overlaps it, combined in a fixed order:
        // the lanes of my head take slots in turn, then fold across those lanes
        const long long n = walk.u_end - walk.u_start;
        const int C = p.num_ctas;
        const int cf = qda_cta_of(T, C, walk.u_start);
        const int ns = qda_cta_of(T, C, walk.u_start + n - 1) - cf + 1;
        const bool maybe_empty = T / C < 8;
        float M = -INFINITY, den = 0.f;
        for (int k = lane >> LOG_NH; k < ns; k += 32 >> LOG_NH) {
          const int c = cf + k;
          if (maybe_empty && qda_cta_row(T, C, c) == qda_cta_row(T, C, c + 1)) continue;
          if (!in_bounds(c + walk.unit < C + p.B * p.Hkv, p.err)) continue;
          const float2 ml = p.part_ml[(size_t)(c + walk.unit) * p.heads_pad + hc * NH + my_h];
          const float mn = fmaxf(M, ml.x);
          den = den * ex2(M - mn) + ml.y * ex2(ml.x - mn);
          M = mn;
        }
#pragma unroll
        for (int off = NH; off < 32; off <<= 1) {
          const float Mo = __shfl_xor_sync(0xffffffffu, M, off);
          const float Do = __shfl_xor_sync(0xffffffffu, den, off);
          const float mn = fmaxf(M, Mo);
          den = (M == -INFINITY ? 0.f : den * ex2(M - mn)) + (Mo == -INFINITY ? 0.f : Do * ex2(Mo - mn));
          M = mn;
        }
        m_run = M;
        inv_den = 1.f / den;
      }
    }

    const bool ok = mbar_wait_bounded(&full[stage], phase, abort_flag, p.err, 1u);
    // one block of R rows of the chunk (FULL) or its last, shorter block: a full block's row indexes are constants
    auto block = [&](auto full_tag, const long long b0, const int rows_in) {
      constexpr bool FULL = decltype(full_tag)::value;
      const int rows_valid = FULL ? R : rows_in;
      const unsigned char* st = smem + L.stage0 + (size_t)stage * L.stage_bytes;
      const int lr0 = (int)(b0 - t0);                       // block's first row within the stage
      // the block's rows [lr0, lr0 + rows_valid) lie in the stage (loads past rows_valid clamp to its last row)
      if (!in_bounds(lr0 >= 0 && rows_valid > 0 && lr0 + rows_valid <= TILE, p.err)) return;
      const uint32_t* sK = reinterpret_cast<const uint32_t*>(st) + (size_t)lr0 * W;
      const uint32_t* sV = reinterpret_cast<const uint32_t*>(st + L.codes_bytes) + (size_t)lr0 * W;
      const uint16_t* sKS = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes) + lr0 * NG;
      const uint16_t* sKB = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes + L.sc_bytes) + lr0 * NG;
      [[maybe_unused]] const uint16_t* sVS = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes + 2 * L.sc_bytes) + lr0 * NG;
      [[maybe_unused]] const uint16_t* sVB = reinterpret_cast<const uint16_t*>(st + 2 * L.codes_bytes + 3 * L.sc_bytes) + lr0 * NG;

      // ---- phase 0: per-(row, group) coefficients of K and V (a fixed trip count, so all the loads issue at once).
      // Blocks with more (row, group) pairs than lanes take two groups of a row per lane and load (NG is even and a
      // row's scales start on a 4-byte boundary); smaller ones one pair per lane.
      constexpr bool PAIRS = R * NG > 32;
      constexpr int P0 = PAIRS ? (R * NG / 2 + 31) / 32 : 1;
#pragma unroll
      for (int it = 0; it < P0 && !PAIRS; ++it) {
        const int idx = lane + 32 * it;
        if (idx < rows_valid * NG) {
          const float2 ak = coeffs<BITS, EXACT_K>(half_bits_to_float_rt(sKS[idx], f16), half_bits_to_float_rt(sKB[idx], f16));
          reinterpret_cast<float4*>(sAB)[idx] = make_float4(ak.x, ak.x, ak.y, ak.y);
          if constexpr (!STATS) {
            const float2 av = coeffs<BITS, EXACT>(half_bits_to_float_rt(sVS[idx], f16), half_bits_to_float_rt(sVB[idx], f16));
            sAV[idx] = av.x;
            sBV[idx] = av.y;
          }
        }
      }
#pragma unroll
      for (int it = 0; it < P0 && PAIRS; ++it) {
        const int i2 = lane + 32 * it;   // groups 2 * i2 and 2 * i2 + 1 of the block's flattened (row, group) list
        if (i2 < rows_valid * (NG / 2)) {
          float2 A, B;
          coeffs2<BITS, EXACT_K>(half2_bits_to_float2_rt(reinterpret_cast<const uint32_t*>(sKS)[i2], f16),
                                 half2_bits_to_float2_rt(reinterpret_cast<const uint32_t*>(sKB)[i2], f16), A, B);
          reinterpret_cast<float4*>(sAB)[2 * i2] = make_float4(A.x, A.x, B.x, B.x);
          reinterpret_cast<float4*>(sAB)[2 * i2 + 1] = make_float4(A.y, A.y, B.y, B.y);
          if constexpr (!STATS) {
            coeffs2<BITS, EXACT>(half2_bits_to_float2_rt(reinterpret_cast<const uint32_t*>(sVS)[i2], f16),
                                 half2_bits_to_float2_rt(reinterpret_cast<const uint32_t*>(sVB)[i2], f16), A, B);
            reinterpret_cast<float2*>(sAV)[i2] = A;
            reinterpret_cast<float2*>(sBV)[i2] = B;
          }
        }
      }
      __syncwarp();

      // ---- phase 1: K partial dots, NH heads x S steps per lane
      float v[NV];
#pragma unroll
      for (int s = 0; s < S; ++s) {
        const int r = min(s * RPS + khalf, rows_valid - 1);
        uint32_t w[KW];
        load_words<KW>(sK + r * W + klane * KW, w);
        float2 f[EK / 2];
        unpack_words<BITS, EXACT_K, KW>(w, f);
        const float4 ab = reinterpret_cast<const float4*>(sAB)[r * NG + gk];
#pragma unroll
        for (int h = 0; h < NH; h += 2) {
          // one chain of EK/2 packed FMAs per head (the unrolled steps and heads give the ILP)
          float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < EK / 2; ++k) {
            a0 = __ffma2_rn(f[k], qk[h][k], a0);
            a1 = __ffma2_rn(f[k], qk[h + 1][k], a1);
          }
          const float2 sums = make_float2(a0.x + a0.y, a1.x + a1.y);
          const float2 part = __ffma2_rn(make_float2(ab.x, ab.y), sums,
                                         __fmul2_rn(make_float2(ab.z, ab.w), make_float2(qs[h], qs[h + 1])));
          v[h * S + s] = part.x;
          v[(h + 1) * S + s] = part.y;
        }
      }

      // ---- phase 2: transposed butterfly over the LK lanes of a K row
#pragma unroll
      for (int k = 0; k < LOG_LK; ++k) {
        const int n = NV >> k;
        const bool upper = (lane >> k) & 1;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float a = v[i], b = v[i + n / 2];
          const float send = upper ? a : b;
          const float keep = upper ? b : a;
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << k);
        }
      }

      // ---- phase 3: block softmax for my head over my rows (the first `seen` rows of the block are visible to it)
      int seen = rows_valid;
      if constexpr (MULTI) {
        const long long vis = walk.u_end - my_hide - b0;
        seen = vis < rows_valid ? (int)max(vis, 0LL) : rows_valid;
      }
      float sc[NVL];
      int rr[NVL];
      bool vis[NVL];   // row rr[i] is in the block and visible to my head (always, in a full single-position block)
      float bm = -INFINITY;
#pragma unroll
      for (int i = 0; i < NVL; ++i) {
        rr[i] = my_s[i] * RPS + khalf;
        float si = v[i];
        if constexpr (COMPAT) si = round_to_input(si, f16) * LOG2E;   // natural units, rounded, then log2 units
        vis[i] = (FULL && !MULTI) || rr[i] < seen;
        sc[i] = vis[i] ? si : -INFINITY;
        bm = fmaxf(bm, sc[i]);
      }
      // lazy rescaling: the reference max m_run of a head moves only when one of its scores exceeds it by more than
      // 8 (a factor 2^8 in the weights), so most blocks skip the cross-lane max and the rescale; the partial keeps
      // (m_run, sum, o) consistent whatever reference it ends with
      const bool moved = !APPLY && __any_sync(0xffffffffu, bm > m_run + 8.f);
      float alpha = 1.f;
      if (moved) {
#pragma unroll
        for (int off = NH; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
        const float m_new = fmaxf(m_run, bm);
        if constexpr (MULTI) {
          alpha = m_new == -INFINITY ? 1.f : ex2(m_run - m_new);   // a head with nothing visible yet keeps 0
        } else {
          alpha = ex2(m_run - m_new);
        }
        m_run = m_new;
        if constexpr (!STATS) {
#pragma unroll
          for (int g = 0; g < NG; ++g) pb[g] *= alpha;
        }
        l_run *= alpha;
      }
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < NVL; ++i) {
        float2* ps = reinterpret_cast<float2*>(sPS) + 2 * (rr[i] * PS_ROW + (my_h >> 1) * NG) + (my_h & 1);
        if constexpr (STATS) {
          if (vis[i]) psum += ex2(sc[i] - m_run);
          continue;
        }
        if (vis[i]) {
          float pr = ex2(sc[i] - m_run);
          if constexpr (APPLY) pr = round_to_input(pr * inv_den, f16);   // normalised, rounded to the input dtype
          psum += pr;
          const float* av = sAV + rr[i] * NG;
          const float* bv = sBV + rr[i] * NG;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const float x = pr * av[g];
            ps[2 * g] = make_float2(x, x);
            pb[g] = fmaf(pr, bv[g], pb[g]);
          }
        } else {   // rows past the chunk (or hidden from the head) take part in the V loop with weight 0
#pragma unroll
          for (int g = 0; g < NG; ++g) ps[2 * g] = make_float2(0.f, 0.f);
        }
      }
      l_run += psum;
      __syncwarp();

      // ---- phase 4: V accumulation (none in pass A)
      if constexpr (STATS) return;
      if (moved) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float a = __shfl_sync(0xffffffffu, alpha, head_lane[h]);
#pragma unroll
          for (int k = 0; k < EV / 2; ++k) o[h][k] = __fmul2_rn(o[h][k], make_float2(a, a));
        }
      }
      const float4* psv = reinterpret_cast<const float4*>(sPS) + gv;
#pragma unroll
      for (int rs = 0; rs < R / VR; ++rs) {
        const int r = rs * VR + vrow;
        uint32_t w[VW];
        load_words<VW>(sV + min(r, rows_valid - 1) * W + vlane * VW, w);
        float2 f[EV / 2];
        unpack_words<BITS, EXACT, VW>(w, f);
        const float4* pr = psv + r * PS_ROW;
#pragma unroll
        for (int h = 0; h < NH; h += 2) {
          const float4 pp = pr[(h / 2) * NG];   // (p A_v, p A_v) of heads h and h + 1
#pragma unroll
          for (int k = 0; k < EV / 2; ++k) {
            o[h][k] = __ffma2_rn(make_float2(pp.x, pp.y), f[k], o[h][k]);
            o[h + 1][k] = __ffma2_rn(make_float2(pp.z, pp.w), f[k], o[h + 1][k]);
          }
        }
      }
      __syncwarp();
    };
    // the chunk's rows are dealt to the warps in blocks of R
    for (long long b0 = c0 + (long long)warp * R; ok && b0 < c1; b0 += (long long)NW * R) {
      const int rows = (int)min((long long)R, c1 - b0);
      // the full-block copy pays with 4 heads per CTA (shorter blocks, more of the work in row indexing); with 2 the
      // larger code is slower
      if (NH == 4 && rows == R) {
        block(std::true_type{}, b0, rows);
      } else {
        block(std::false_type{}, b0, rows);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);

    if (c1 == walk.u_end || c1 == r1) {
      // ------------------------------------------------------------- end of a segment
      // l and the p * B_v sums: over all lanes owning the same head
#pragma unroll
      for (int off = NH; off < 32; off <<= 1) {
        l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
        if constexpr (!STATS) {
#pragma unroll
          for (int g = 0; g < NG; ++g) pb[g] += __shfl_xor_sync(0xffffffffu, pb[g], off);
        }
      }
      if constexpr (!STATS && VR > 1) {
        // the lanes of one V slice took different rows: add their sums (every lane then holds the slice's total)
#pragma unroll
        for (int off = VL; off < 32; off <<= 1)
#pragma unroll
          for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int k = 0; k < EV / 2; ++k)
              o[h][k] = __fadd2_rn(o[h][k], make_float2(__shfl_xor_sync(0xffffffffu, o[h][k].x, off),
                                                        __shfl_xor_sync(0xffffffffu, o[h][k].y, off)));
      }
      if constexpr (!STATS) {
        if (lane < NH) {   // lane < NH owns head my_h; all heads are covered once
#pragma unroll
          for (int g = 0; g < NG; ++g) sPB[my_h * NG + g] = pb[g];
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float b = sPB[h * NG + gv];
#pragma unroll
          for (int k = 0; k < EV / 2; ++k) o[h][k] = __fadd2_rn(o[h][k], make_float2(b, b));
        }
      }
      named_barrier_sync(1, NW * 32);   // every warp is done with its scratch before it becomes the combine area
      if constexpr (!STATS) {
        if (vrow == 0) {
#pragma unroll
          for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int k = 0; k < EV / 2; ++k)
              reinterpret_cast<float2*>(comb_o + (warp * NH + h) * D + vlane * EV)[k] = o[h][k];
        }
      }
      if (lane < NH) {
        comb_m[warp * NH + my_h] = m_run;
        comb_l[warp * NH + my_h] = l_run;
      }
      named_barrier_sync(1, NW * 32);
      const long long slot = (long long)cta + walk.unit;
      // pass A writes only (max, sum) per head; pass B only o (its weights are already normalised, and other CTAs
      // of pass B may still be reading pass A's statistics)
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
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
}

// DSET 0: D in {64, 128}; 1: D in {256, 512} (two translation units per (bits, exact), compiled in parallel)
template <int BITS, bool EXACT, int MODE, int DSET, typename Fn>
cudaError_t with_split2_kernel_m(int D, int nh, int ng, Fn&& f) {
#define QDA_V2(D_, NH_, NG_) \
  if (D == D_ && nh == NH_ && ng == NG_) return f(qda_split2_kernel<BITS, D_, NH_, NG_, EXACT, MODE>);
  if constexpr (DSET == 0) {
    QDA_V2(64, 2, 1) QDA_V2(64, 2, 2) QDA_V2(64, 4, 1) QDA_V2(64, 4, 2)
    QDA_V2(128, 2, 1) QDA_V2(128, 2, 2) QDA_V2(128, 2, 4) QDA_V2(128, 4, 1) QDA_V2(128, 4, 2) QDA_V2(128, 4, 4)
  } else {
    QDA_V2(256, 2, 2) QDA_V2(256, 2, 4) QDA_V2(256, 2, 8)
    QDA_V2(256, 4, 2) QDA_V2(256, 4, 4) QDA_V2(256, 4, 8)
    QDA_V2(512, 2, 4) QDA_V2(512, 2, 8) QDA_V2(512, 2, 16)
  }
#undef QDA_V2
  return cudaErrorInvalidValue;
}

template <int BITS, bool EXACT, int DSET, typename Fn>
cudaError_t with_split2_kernel(int D, int nh, int ng, int mode, Fn&& f) {
  switch (mode) {
    case 0: return with_split2_kernel_m<BITS, EXACT, 0, DSET>(D, nh, ng, f);
    case 1: return with_split2_kernel_m<BITS, EXACT, 1, DSET>(D, nh, ng, f);
    case 2: return with_split2_kernel_m<BITS, false, 2, DSET>(D, nh, ng, f);   // pass A reads no V: no exact variant
    case 3: return with_split2_kernel_m<BITS, EXACT, 3, DSET>(D, nh, ng, f);
    default: return cudaErrorInvalidValue;
  }
}

template <int BITS, bool EXACT, int DSET>
cudaError_t launch_split2(const QdaParams& p, int D, int nh, int ng, dim3 grid, size_t smem, cudaStream_t s) {
  return with_split2_kernel<BITS, EXACT, DSET>(D, nh, ng, p.mode, [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_limit(kern, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, QDA_THREADS, smem, s, p.launch_pdl != 0, p);
  });
}

template <int BITS, bool EXACT, int DSET>
cudaError_t occupancy_split2(int D, int nh, int ng, size_t smem, int* n) {
  // both instances of a shape have the same resources; the single-query one stands for both
  return with_split2_kernel<BITS, EXACT, DSET>(D, nh, ng, 0, [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_limit(kern, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, QDA_THREADS, smem);
  });
}

}  // namespace qda
