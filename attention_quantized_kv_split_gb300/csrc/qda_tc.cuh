// Tensor-core split kernel of quantized-KV decode attention for 4-bit codes (sm_103a): the q . K contraction of
// every 128-row tile runs on tcgen05 with the codes as exact 16-bit operands; the softmax and the V side stay on
// the CUDA cores in fp32.
//
// The block structure is the flash-decoding split-N of mlx-bun fused-decode-kernel.ts (BLOCK_SOURCE: per-block
// running max / sum-exp / unnormalised o, merged later by MERGE_SOURCE) over one contiguous row range per CTA
// (qda_split.cuh). What is new is where the score dot product runs. With four query heads per KV head and 4-bit
// codes, a CUDA-core kernel spends most of its issue slots on the scores (unpacking, 4 x D FMAs, a cross-lane
// reduction); here a row's codes are turned into sixteen-bit values and the tensor cores do the sums:
//   * a 4-bit code c becomes the bf16 (or fp16) value 128 + c (1024 + c): one AND/OR per two codes, exact;
//   * the factored dot of the SCORE_ROW comment, s * sum_g(c q) + b * sum_g(q), is taken per group g of GS
//     codes: one MMA chain per group writes sum_{d in g} (OFF + c_d) q_d for the CTA's four heads into its own
//     16 accumulator columns (M = 128 rows, N = 16 with heads 4..15 zero, K = 16 per instruction, fp32 sums),
//     and the epilogue forms s * acc + (b - OFF * s) * sum_g(q) in fp32;
//   * the A operand (the codes) goes from the registers straight into tensor memory, the B operand (q of the
//     unit, its own 16-bit values, exact) sits in shared memory.
// One thread issues a tcgen05 MMA about every 50 cycles whatever its N up to 128, so a tile's D / 16 MMAs take a
// fixed time to issue; two issuing warps halve it, and every stage runs in its own warps, linked by mbarriers, so
// that pipeline step i + 1 is converted and multiplied while step i's scores and step i - 1's V rows are worked on.
// A step is one 128-row tile at D = 256 and two at D = 128 (both fit in tensor memory double-buffered; the per-step
// waits and bookkeeping are then paid once per 256 rows):
//   warps 0-3   converters: K codes of a step's tiles (lane quarter w: rows 32 w .. 32 w + 31 of each tile) ->
//               tensor memory (A), and at a new (sequence, KV head) the unit's q into the B operand and its
//               per-group sums (loaded before the chunk's K slot is waited for, so the two overlap);
//   warps 4-7   epilogue: accumulators of their lane quarter -> scores, the online softmax (reference max per
//               quarter and head), p * A_v per (row, group) for the V warps, sums of p and of p * B_v;
//   warps 8-15  V: 16 rows per tile of each step (consecutive rows), all four heads, packed fp32 FMAs on the CUDA
//               cores (codes as 0.5 + c / 256, or 0.5 + c / 32 for fp32 outputs);
//   warp 16     producer: 2-D tensor copies of the K tiles (their 128-byte swizzle lets one thread per row read its
//               row without bank conflicts) into one ring, 1-D bulk copies of the V codes, scales and biases into
//               a second;
//   warps 17-18 issue the MMAs of even and odd steps (double-buffered A operand and accumulators in tensor
//               memory, which warp 17 allocates and frees).
// Every wait is bounded; after a timeout every warp still passes every barrier (with no work), so the kernel
// always returns and frees its tensor memory.
#pragma once

#include <cuda.h>

#include "qda_split2.cuh"

namespace qda {

__host__ __device__ constexpr int tc_tmem_cols(int used) {
  return used <= 32 ? 32 : used <= 64 ? 64 : used <= 128 ? 128 : used <= 256 ? 256 : 512;
}

// Bounded wait on a barrier phase taken by lane 0, its result shared with the warp (warp-uniform control flow).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort, err, 1u);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The V codes of chunk [c0, c1) of the tile starting at row t0 and the 8-row aligned cover of its scales and biases
// into V-ring slot `vst`, completing on `full`. Called by the producer warp.
__device__ __forceinline__ void tc_issue_v(const QdaParams& p, unsigned char* vst, const QdaTcLayout& L,
                                           uint64_t* full, long long c0, long long c1, long long t0, long long T,
                                           uint64_t pol) {
  const int lane = threadIdx.x & 31;
  const int NG = p.NG;
  const uint32_t RB = p.W * 4, SB = NG * 2;
  const uint32_t cbytes = (uint32_t)(c1 - c0) * RB;
  const size_t coff = (size_t)(c0 - t0) * RB;
  const long long s0 = c0 & ~7LL;
  const long long s1 = min((c1 + 7) & ~7LL, T);
  const uint32_t sbytes = (uint32_t)(s1 - s0) * SB;
  const uint32_t s16 = sbytes & ~15u;
  const size_t soff = (size_t)(s0 - t0) * SB;
  unsigned char* sc = vst + L.v_bytes;
  const bool inb = in_bounds(c0 >= t0 && c0 < c1 && c1 <= T && c1 - t0 <= L.slot_rows && s1 <= T && s0 >= t0 &&
                                 coff + cbytes <= L.v_bytes && soff + sbytes <= L.sc_bytes,
                             p.err);
  if (lane == 0 && !inb) mbar_arrive_expect_tx(full, 0);
  if (!inb) return;
  if (lane == 0) {
    if (s16 != sbytes) {   // a ragged last < 16 bytes of the scale arrays: plain loads, published by the arrive
      const uint16_t* srcs[4] = {p.ks, p.kb, p.vs, p.vb};
      for (int a = 0; a < 4; ++a) {
        const uint16_t* src = srcs[a] + s0 * NG + s16 / 2;
        uint16_t* dst = reinterpret_cast<uint16_t*>(sc + a * L.sc_bytes + soff + s16);
        for (uint32_t k = 0; k < (sbytes - s16) / 2; ++k) dst[k] = src[k];
      }
    }
    mbar_arrive_expect_tx(full, cbytes + 4 * s16);
  }
  __syncwarp();
  if (lane == 0) {
    bulk_g2s(vst + coff, p.vp + c0 * p.W, cbytes, full, pol);
  } else if (lane < 5 && s16) {
    const int a = lane - 1;
    const uint16_t* src = a == 0 ? p.ks : a == 1 ? p.kb : a == 2 ? p.vs : p.vb;
    bulk_g2s(sc + a * L.sc_bytes + soff, src + s0 * NG, s16, full, pol);
  }
}

// A row's NG 16-bit scale or bias values (NG * 2 bytes, aligned to that size) in one shared-memory load: value g
// is half g & 1 of word g / 2.
template <int NG>
__device__ __forceinline__ void load_halves(const uint16_t* src, uint32_t (&w)[(NG + 1) / 2]) {
  if constexpr (NG == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (NG == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    w[0] = v.x; w[1] = v.y;
  } else {
    static_assert(NG == 2, "2, 4 or 8 groups");
    w[0] = *reinterpret_cast<const uint32_t*>(src);
  }
}
__device__ __forceinline__ uint32_t half_of(const uint32_t* w, int g) {
  return (w[g >> 1] >> (16 * (g & 1))) & 0xFFFFu;
}

// Input dtype of q, scales and biases: DT = 0 bf16, 1 fp16 (compile-time: one instruction per conversion), 2 chosen
// at run time from p.f16 (the D = 256 instances: measured faster there, the compile-time form 5-7 % slower; at
// D = 128 it is 6 % faster).
template <int DT>
__device__ __forceinline__ float tc_half_to_float(uint32_t u16, bool f16) {
  if constexpr (DT == 2) {
    return half_bits_to_float_rt(u16, f16);
  } else {
    return half_bits_to_float<DT == 1>(u16);
  }
}

// V codes as floats, per output form. 16-bit outputs: 0.5 + c / 256 (a byte permute per code). fp32 outputs:
// 0.5 + c / 32 -- each code shifted into bits 3..6 of its byte, then a byte permute under the exponent byte 0x3F --
// so that the code, not the offset 0.5, carries most of each value (a sum of w * (0.5 + c / 32) rounds about twice
// as coarsely as the code part alone, against 18 times for c / 256): two shifts and masks per word plus one permute
// per code, 3 instructions per word fewer than exact codes (2^23 + c minus 2^23).
template <bool FP32OUT, int NW>
__device__ __forceinline__ void tc_unpack_v(const uint32_t (&w)[NW], float2 (&f)[NW * 4]) {
  if constexpr (FP32OUT) {
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      const uint32_t lo = (w[k] << 3) & 0x78787878u;   // codes 0, 2, 4, 6 at bits 3..6 of bytes 0..3
      const uint32_t hi = (w[k] >> 1) & 0x78787878u;   // codes 1, 3, 5, 7
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t sel = 0x7054u | ((uint32_t)j << 8);   // bytes [0, 0, code << 3, 0x3F]
        f[4 * k + j] = make_float2(__uint_as_float(__byte_perm(lo, 0x3F000000u, sel)),
                                   __uint_as_float(__byte_perm(hi, 0x3F000000u, sel)));
      }
    }
  } else {
    unpack_words<4, false, NW>(w, f);
  }
}
// s * c + b = A * f + B for the code form above: c = 32 f - 16 (fp32 outputs), c = 256 f - 128 (16-bit outputs).
template <bool FP32OUT>
__device__ __forceinline__ float2 tc_coeffs_v(float s, float b) {
  if constexpr (FP32OUT) {
    return make_float2(32.0f * s, fmaf(-16.0f, s, b));
  } else {
    return coeffs<4, false>(s, b);
  }
}

template <int D, int NH, int NG, bool FP32OUT, int DT>
__global__ void __launch_bounds__(QDA_TC_THREADS, 1)
    qda_tc_kernel(const __grid_constant__ QdaParams p, const __grid_constant__ CUtensorMap tmk) {
  constexpr int TILE = QDA_TC_TILE;
  constexpr int RB = D / 2, W = D / 8, CPR = RB / 16, GS = D / NG;
  constexpr int SLOT = QDA_TC_SLOT_BYTES / RB;   // rows per ring slot: SLOT / TILE MMA tiles
  constexpr int BOXW = RB >= 128 ? 128 : RB;     // bytes per row of one tensor-copy box (its rows: <= 256)
  constexpr int BOXES_Y = SLOT / 256, BOXES_X = RB / BOXW;
  constexpr int EV = D >= 256 ? D / 32 : 8, VL = D / EV, VR = 32 / VL, VW = EV / 8;
  constexpr int A_COLS = D / 2, ACC_COLS = 16 * NG;
  // rows per pipeline step: two MMA tiles at D = 128 (both tiles' A operands and accumulators, double-buffered, fit
  // in tensor memory), so every role's per-step waits, arrivals and bookkeeping are paid once per 256 rows
  constexpr int TPS = D == 128 ? 2 : 1, STEP = TPS * TILE;
  constexpr int TMEM_COLS = tc_tmem_cols(2 * TPS * (A_COLS + ACC_COLS));
  constexpr int KSTEPS = D / 16;
  // the V loop two rows deep for 16-bit outputs, one for fp32 outputs; the conversion loop not unrolled (smaller
  // code: the roles share each sub-partition's instruction cache) -- each measured faster
  constexpr int V_UNROLL = FP32OUT ? 1 : 2;
  // the epilogue loads its accumulators in NSPLIT runs of NGH groups (8 groups: two runs, against spills)
  constexpr int NSPLIT = NG == 8 ? 2 : 1, NGH = NG / NSPLIT;
  // the epilogue's per-group score and weight updates as packed f32x2 operations (heads in pairs) up to 4 groups
  // per row: measured 1 % faster there, 2.5 % slower at 8 groups
  constexpr bool PAIRED = NG <= 4;
  constexpr int EPI0 = QDA_TC_CONV, V0 = EPI0 + QDA_TC_EPI, PRODUCER = V0 + QDA_TC_VW, MMA_WARP = PRODUCER + 1;
  // MMA_WARP issues the MMAs of even steps and allocates tensor memory, MMA_WARP + 1 those of odd steps
  constexpr int EV_THREADS = (QDA_TC_EPI + QDA_TC_VW) * 32;
  static_assert(NH == 4, "four query heads per CTA");
  static_assert(NG >= 2 && GS >= 32 && GS % 16 == 0, "two or more groups of at least 32 codes per row");
  static_assert(2 * TPS * (A_COLS + ACC_COLS) <= 512, "tensor memory");
  static_assert(RB == 64 || RB % 128 == 0, "K rows of 64 or 128k bytes");
  static_assert(SLOT % 256 == 0 && BOXES_X == 1, "slots of whole 256-row boxes, one box column");
  static_assert(QDA_TC_VW * 16 == TILE && QDA_TC_CONV * 32 == TILE && QDA_TC_EPI * 32 == TILE && SLOT % STEP == 0,
                "warp shares");

  extern __shared__ __align__(1024) unsigned char smem[];
  const int KS = p.kstages, VS = p.stages;
  const QdaTcLayout Ls = qda_tc_layout(D, NH, NG, KS, VS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* kfull = bars;          // [KS <= 8] K slot landed
  uint64_t* kempty = bars + 8;     // [KS] K slot converted (4 converter warps)
  uint64_t* vfull = bars + 16;     // [VS <= 12] V codes and scales landed
  uint64_t* vempty = bars + 28;    // [VS] scales and V rows of every tile of the slot used (4 epilogue + 8 V warps)
  uint64_t* a_full = bars + 40;    // [2] A buffer written (4 converter warps)
  uint64_t* a_free = bars + 42;    // [2] the MMAs that read A buffer b are complete
  uint64_t* acc_full = bars + 44;  // [2] accumulator buffer b holds the tile's sums
  uint64_t* acc_empty = bars + 46; // [2] accumulator buffer b read (4 epilogue warps)
  uint64_t* p_full = bars + 48;    // [2] p * A_v buffer b written (4 epilogue warps)
  uint64_t* p_empty = bars + 50;   // [2] p * A_v buffer b read (8 V warps)
  uint64_t* qs_full = bars + 52;   // [2] B operand and q sums of unit parity b written (4 converter warps)
  uint64_t* qs_free = bars + 54;   // [2] q sums of unit parity b no longer read (4 epilogue warps)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 480);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 484);
  unsigned char* b_op = smem + Ls.b_op;
  float* qs_all = reinterpret_cast<float*>(smem + Ls.qs);
  float* alpha_s = reinterpret_cast<float*>(smem + Ls.alpha);
  float4* ps = reinterpret_cast<float4*>(smem + Ls.ps);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x / p.head_chunks, hc = blockIdx.x - cta * p.head_chunks;
  const long long T = p.total_rows;
  const long long r0 = qda_cta_row_fast(T, p.num_ctas, p.cta_magic, cta);
  const long long r1 = qda_cta_row_fast(T, p.num_ctas, p.cta_magic, cta + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], QDA_TC_CONV);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], QDA_TC_EPI + QDA_TC_VW);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&a_full[k], QDA_TC_CONV);
      mbar_init(&a_free[k], 1);
      mbar_init(&acc_full[k], 1);
      mbar_init(&acc_empty[k], QDA_TC_EPI);
      mbar_init(&p_full[k], QDA_TC_EPI);
      mbar_init(&p_empty[k], QDA_TC_VW);
      mbar_init(&qs_full[k], QDA_TC_CONV);
      mbar_init(&qs_free[k], QDA_TC_EPI);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) tmem_alloc(tmem_slot, TMEM_COLS);
  // B operand rows (heads) 4..15 of both buffers stay zero for the whole kernel
  for (int k = threadIdx.x; k < 4 * D; k += QDA_TC_THREADS) reinterpret_cast<uint4*>(b_op)[k] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // launched with programmatic dependent launch: everything above is CTA-local; the grid before this one on the
  // stream is complete and visible from here on
  pdl_wait();
  pdl_launch_dependents();

  if (r0 < r1) {
    ChunkWalker walk;   // chunks: a slot of SLOT rows intersected with one (sequence, KV head) and the CTA's range
    walk.init(p, r0, r1);
    long long c0, c1, t0;
    const bool f16 = DT == 2 ? p.f16 != 0 : DT == 1;
    // the steps of a slot that a chunk [c0, c1) (slot rows lr0 .. lr1) touches: st0 .. st1 - 1
    auto tiles_of = [](int lr0, int lr1, int& st0, int& st1) {
      st0 = lr0 / STEP;
      st1 = (lr1 + STEP - 1) / STEP;
    };

    if (warp == PRODUCER) {
      // ---------------------------------------------------------------------------------- producer warp
      const uint64_t pol = policy_evict_first();
      int i = 0, ks = 0, kph = 0, vs = 0, vph = 0;
      while (walk.next(p, c0, c1, t0)) {
        if (blockIdx.x == 0 && i == p.stall_chunk) break;   // testing aid: the consumers' wait for it must run out
        if (i >= KS && !wait_warp(&kempty[ks], kph ^ 1, abort_flag, p.err)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&kfull[ks], (uint32_t)Ls.k_bytes);
          unsigned char* kst = smem + Ls.k0 + (size_t)ks * Ls.k_bytes;
          for (int by = 0; by < BOXES_Y; ++by)   // the whole slot: rows past the cache read as zero
            tma_load_2d(kst + (size_t)by * 256 * BOXW, &tmk, 0, (int)t0 + 256 * by, &kfull[ks], pol);
        }
        __syncwarp();
        if (i >= VS && !wait_warp(&vempty[vs], vph ^ 1, abort_flag, p.err)) break;
        tc_issue_v(p, smem + Ls.v0 + (size_t)vs * Ls.vstage_bytes, Ls, &vfull[vs], c0, c1, t0, T, pol);
        ++i;
        if (++ks == KS) {
          ks = 0;
          kph ^= 1;
        }
        if (++vs == VS) {
          vs = 0;
          vph ^= 1;
        }
      }
      if (lane == 0) {   // every issued copy lands before the CTA exits
        for (int j = (i > KS ? i - KS : 0); j < i; ++j) mbar_wait_drain(&kfull[j % KS], (j / KS) & 1, p.err);
        for (int j = (i > VS ? i - VS : 0); j < i; ++j) mbar_wait_drain(&vfull[j % VS], (j / VS) & 1, p.err);
      }
      __syncwarp();
    } else if (warp >= MMA_WARP) {
      // ---------------------------------------------------------------------------------- MMA warps
      // Two issuers, one per A / accumulator buffer (step parity): one thread issues an MMA about every 50
      // cycles, and two threads keep the tensor pipe twice as busy.
      const int ab = warp - MMA_WARP;
      const uint32_t idesc = mma_idesc_f16(TILE, 16, f16);
      // descriptor of K step 0 of B buffer 0; step s of buffer u adds (u * 32 D + 512 s) / 16 to the address field
      const uint64_t bdesc0 = smem_desc_kmajor(smem_addr(b_op), 256, 128);
      const uint32_t a0 = tbase + ab * TPS * A_COLS;
      const uint32_t d0 = tbase + 2 * TPS * A_COLS + ab * TPS * ACC_COLS;
      int j = 0, uidx = -1, cur_unit = -1, issued = -1;
      bool go = true;
      while (go && walk.next(p, c0, c1, t0)) {
        if (walk.unit != cur_unit) {
          cur_unit = walk.unit;
          ++uidx;
        }
        int st0, st1;
        tiles_of((int)(c0 - t0), (int)(c1 - t0), st0, st1);
        for (int st = st0; st < st1; ++st, ++j) {
          if ((j & 1) != ab) continue;
          if (!wait_warp(&a_full[ab], (j >> 1) & 1, abort_flag, p.err) ||
              (j >= 2 && !wait_warp(&acc_empty[ab], ((j >> 1) - 1) & 1, abort_flag, p.err))) {
            go = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint64_t bd = bdesc0 + (uint64_t)((uidx & 1) * 2 * D);
#pragma unroll
            for (int t = 0; t < TPS; ++t) {
#pragma unroll
              for (int s = 0; s < KSTEPS; ++s) {
                // K step s covers codes of group (16 s) / GS; the group's first step starts its accumulator afresh
                mma_f16_ts(d0 + t * ACC_COLS + 16 * ((16 * s) / GS), a0 + t * A_COLS + 8 * s, bd + (uint64_t)(32 * s),
                           idesc, (16 * s) % GS != 0);
              }
            }
            mma_commit(&a_free[ab]);
            mma_commit(&acc_full[ab]);
          }
          __syncwarp();
          issued = j;
        }
      }
      // every MMA this warp issued is complete before the tensor memory is freed
      if (issued >= 0 && lane == 0) mbar_wait_drain(&a_free[ab], (issued >> 1) & 1, p.err);
      __syncwarp();
    } else if (warp < EPI0) {
      // ---------------------------------------------------------------------------------- converter warps
      const uint32_t tl = tbase + ((uint32_t)(32 * warp) << 16);
      const uint32_t magic = f16 ? 0x64006400u : 0x43004300u;   // OFF + c in the low mantissa bits
      int i = 0, j = 0, ks = 0, kph = 0, uidx = -1, cur_unit = -1;
      bool ok = true;   // false once a wait of this warp gave up: the warp then passes every barrier with no work
      while (walk.next(p, c0, c1, t0)) {
        if (walk.unit != cur_unit) {
          // a new (sequence, KV head): its q into B operand buffer (unit parity) and its sums per group, once the
          // MMAs that read that buffer (two units back) are complete -- the latest MMA of each A buffer covers
          // every earlier one of its issuer -- and the epilogue is done with those sums
          cur_unit = walk.unit;
          ++uidx;
          const int par = uidx & 1;
          if (j >= 1) ok = ok && wait_warp(&a_free[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.err);
          if (j >= 2) ok = ok && wait_warp(&a_free[j & 1], ((j >> 1) - 1) & 1, abort_flag, p.err);
          if (uidx >= 2) ok = ok && wait_warp(&qs_free[par], ((uidx >> 1) - 1) & 1, abort_flag, p.err);
          if (ok) {
            constexpr int OCT = D / 8;
            const int item = threadIdx.x;   // (head, octet of q): converter threads 0..127
            float sum = 0.f;
            if (item < NH * OCT) {
              const int h = item / OCT, wi = item - h * OCT;
              const int jq = hc * NH + h;
              uint4 a = make_uint4(0, 0, 0, 0);
              if (jq < p.nrep * p.L) {
                const long long row = qda_q_row(walk.b, walk.kvh, jq, p.nrep, p.L, p.H);
                if (in_bounds(row < (long long)p.B * p.L * p.H, p.err))
                  a = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + row * D + 8 * wi);
              }
              // position 2j + e of octet wi holds q[8 wi + j + 4 e]: the order in which the conversion below lays
              // the codes of a word into tensor-memory columns
              const uint4 bw = make_uint4(__byte_perm(a.x, a.z, 0x5410), __byte_perm(a.x, a.z, 0x7632),
                                          __byte_perm(a.y, a.w, 0x5410), __byte_perm(a.y, a.w, 0x7632));
              *reinterpret_cast<uint4*>(b_op + par * 32 * D + wi * 256 + (h >> 3) * 128 + (h & 7) * 16) = bw;
              const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
              for (int k = 0; k < 4; ++k)
                sum += tc_half_to_float<DT>(u[k] & 0xFFFFu, f16) + tc_half_to_float<DT>(u[k] >> 16, f16);
            }
#pragma unroll
            for (int off = 1; off < GS / 8; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (item < NH * OCT) {
              const int h = item / OCT, wi = item - h * OCT;
              if ((wi & (GS / 8 - 1)) == 0) qs_all[par * NG * NH + (wi / (GS / 8)) * NH + h] = sum;
            }
          }
          fence_proxy_async();
          named_barrier_sync(2, QDA_TC_CONV * 32);
          if (lane == 0) mbar_arrive(&qs_full[par]);
        }
        // the chunk's K slot, waited for after a new unit's q loads, so that these overlap its arrival (at the
        // start of a CTA, where the first MMA then comes about 2 us sooner)
        ok = ok && wait_warp(&kfull[ks], kph, abort_flag, p.err);
        int st0, st1;
        tiles_of((int)(c0 - t0), (int)(c1 - t0), st0, st1);
        const unsigned char* sK = smem + Ls.k0 + (size_t)ks * Ls.k_bytes;
        for (int st = st0; st < st1; ++st, ++j) {
          // A buffer j & 1 was last read by the MMAs of step j - 2
          if (j >= 2) ok = ok && wait_warp(&a_free[j & 1], ((j >> 1) - 1) & 1, abort_flag, p.err);
          tc_fence_after();
          for (int t = 0; t < TPS && ok; ++t) {
            const int row = st * STEP + t * TILE + 32 * warp + lane;   // the slot row this thread converts
#pragma unroll 1
            for (int c = 0; c < CPR; ++c) {
              const unsigned char* src;
              if constexpr (RB == 64) {
                src = sK + row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
              } else {
                src = sK + row * 128 + (((c & 7) ^ (row & 7)) << 4);
              }
              const uint4 x = *reinterpret_cast<const uint4*>(src);
              const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
              uint32_t out[16];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                // column 4 w + j of word w holds (code j, code j + 4) of the word as (low, high) halves
                out[4 * t + 0] = (wv[t] & 0x000F000Fu) | magic;
                out[4 * t + 1] = ((wv[t] >> 4) & 0x000F000Fu) | magic;
                out[4 * t + 2] = ((wv[t] >> 8) & 0x000F000Fu) | magic;
                out[4 * t + 3] = ((wv[t] >> 12) & 0x000F000Fu) | magic;
              }
              tmem_st16(tl + ((j & 1) * TPS + t) * A_COLS + 16 * c, out);
            }
          }
          if (ok) tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[j & 1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&kempty[ks]);
        ++i;
        if (++ks == KS) {
          ks = 0;
          kph ^= 1;
        }
      }
    } else {
      // ---------------------------------------------------------------------------- epilogue and V warps
      const bool epi = warp < V0;
      // lane quarter (rows 32 q .. 32 q + 31 of a tile); a V warp's rows lie in one quarter of one tile
      const int q = epi ? warp - EPI0 : TPS == 1 ? (warp - V0) >> 1 : (warp - V0) & 3;
      const int ev_tid = threadIdx.x - EPI0 * 32;
      // End of a segment, after both roles wrote their parts into the chunk's V slot (the combine area; its copies
      // have landed and both roles are done with it): one partial (max, sum, o[D]) per head from the four lane
      // quarters, combined in a fixed order by the 384 epilogue and V threads.
      auto combine = [&](float* co, int unit) {
        const float* cm = co + QDA_TC_VW * NH * D;
        const float* cl = cm + 4 * NH;
        const float* cpb = cl + 4 * NH;
        named_barrier_sync(1, EV_THREADS);
        const long long slot = (long long)cta + unit;
        for (int idx = ev_tid; idx < NH * D; idx += EV_THREADS) {
          const int h = idx / D, d = idx - h * D, g = d / GS;
          float M = -INFINITY;
#pragma unroll
          for (int k = 0; k < 4; ++k) M = fmaxf(M, cm[k * NH + h]);
          float O = 0.f, Lsum = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float mk = cm[k * NH + h];
            const float wt = mk == -INFINITY ? 0.f : ex2(mk - M);
            const float ok4 = co[(2 * k * NH + h) * D + d] + co[((2 * k + 1) * NH + h) * D + d] +
                              cpb[(k * NG + g) * NH + h];
            O = fmaf(wt, ok4, O);
            Lsum = fmaf(wt, cl[k * NH + h], Lsum);
          }
          const size_t hp = (size_t)slot * p.heads_pad + (size_t)hc * NH + h;
          if (!in_bounds(slot < (long long)p.num_ctas + p.B * p.Hkv && hc * NH + h < p.heads_pad, p.err)) continue;
          p.part_o[hp * D + d] = O;
          if (d == 0) p.part_ml[hp] = make_float2(M, Lsum);
        }
        fence_proxy_async();   // these generic writes to the slot come before the copies that refill it
        named_barrier_sync(1, EV_THREADS);
      };
      int i = 0, j = 0, vs = 0, vph = 0;
      bool ok = true;

      if (epi) {
        // ------------------------------------------------------------------------------ epilogue warps
        const uint32_t tl = tbase + ((uint32_t)(32 * q) << 16);
        const float OFF = f16 ? 1024.f : 128.f;
        // reference max, sum of weights and sums of p * B_v over this thread's rows, per head
        float m_run[NH], l_run[NH];
        float pb[NG][NH];
        auto reset = [&]() {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            m_run[h] = -INFINITY;
            l_run[h] = 0.f;
#pragma unroll
            for (int g = 0; g < NG; ++g) pb[g][h] = 0.f;
          }
        };
        reset();
        int uidx = -1, cur_unit = -1;
        while (walk.next(p, c0, c1, t0)) {
          unsigned char* vst = smem + Ls.v0 + (size_t)vs * Ls.vstage_bytes;
          const int lr0 = (int)(c0 - t0), lr1 = (int)(c1 - t0);
          if (walk.unit != cur_unit) {
            cur_unit = walk.unit;
            ++uidx;
            ok = ok && wait_warp(&qs_full[uidx & 1], (uidx >> 1) & 1, abort_flag, p.err);
          }
          const float* qs = qs_all + (uidx & 1) * NG * NH;
          ok = ok && wait_warp(&vfull[vs], vph, abort_flag, p.err);
          const uint16_t* sKS = reinterpret_cast<const uint16_t*>(vst + Ls.v_bytes);
          const uint16_t* sKB = sKS + Ls.sc_bytes / 2;
          const uint16_t* sVS = sKB + Ls.sc_bytes / 2;
          const uint16_t* sVB = sVS + Ls.sc_bytes / 2;
          int st0, st1;
          tiles_of(lr0, lr1, st0, st1);
          for (int st = st0; st < st1; ++st, ++j) {
            const int pbuf = j & 1;
            ok = ok && wait_warp(&acc_full[pbuf], (j >> 1) & 1, abort_flag, p.err);
            tc_fence_after();
            const int m = 32 * q + lane;   // the row this thread scores in each tile of the step
            float sc[TPS][NH];
            bool valid[TPS];
#pragma unroll
            for (int t = 0; t < TPS; ++t) {
              const int row = st * STEP + t * TILE + m;   // its slot row
              valid[t] = row >= lr0 && row < lr1;
#pragma unroll
              for (int h = 0; h < NH; ++h) sc[t][h] = 0.f;
            }
            // the accumulators of NSPLIT runs of groups in turn (two at 8 groups: 16 live values fewer), the buffer
            // released to the MMAs after the last run is loaded
#pragma unroll
            for (int hf = 0; hf < NSPLIT; ++hf) {
              float acc[TPS][NGH][NH];
              if (ok) {
#pragma unroll
                for (int t = 0; t < TPS; ++t)
#pragma unroll
                  for (int gg = 0; gg < NGH; ++gg)
                    tmem_ld<NH>(tl + 2 * TPS * A_COLS + (pbuf * TPS + t) * ACC_COLS + 16 * (hf * NGH + gg), acc[t][gg]);
                tmem_wait_ld();
              } else {
#pragma unroll
                for (int t = 0; t < TPS; ++t)
#pragma unroll
                  for (int gg = 0; gg < NGH; ++gg)
#pragma unroll
                    for (int h = 0; h < NH; ++h) acc[t][gg][h] = 0.f;
              }
              if (hf == NSPLIT - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[pbuf]);
              }
#pragma unroll
              for (int t = 0; t < TPS; ++t) {
                const int row = st * STEP + t * TILE + m;
                uint32_t ksw[NG / 2], kbw[NG / 2];   // a row's scales and biases: one vector load per array
                load_halves<NG>(sKS + row * NG, ksw);
                load_halves<NG>(sKB + row * NG, kbw);
#pragma unroll
                for (int gg = 0; gg < NGH; ++gg) {
                  const int g = hf * NGH + gg;
                  const float s = tc_half_to_float<DT>(half_of(ksw, g), f16);
                  const float b = tc_half_to_float<DT>(half_of(kbw, g), f16);
                  const float S = p.qscale * s;
                  const float Bc = p.qscale * fmaf(-OFF, s, b);
                  const float4 q4 = reinterpret_cast<const float4*>(qs)[g];
                  const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
                  if constexpr (PAIRED) {   // heads in pairs, packed f32x2 (the same roundings)
#pragma unroll
                    for (int h = 0; h < NH; h += 2) {
                      float2 v2 = __ffma2_rn(make_float2(Bc, Bc), make_float2(qv[h], qv[h + 1]),
                                             make_float2(sc[t][h], sc[t][h + 1]));
                      v2 = __ffma2_rn(make_float2(S, S), make_float2(acc[t][gg][h], acc[t][gg][h + 1]), v2);
                      sc[t][h] = v2.x;
                      sc[t][h + 1] = v2.y;
                    }
                  } else {
#pragma unroll
                    for (int h = 0; h < NH; ++h) sc[t][h] = fmaf(S, acc[t][gg][h], fmaf(Bc, qv[h], sc[t][h]));
                  }
                }
              }
            }
            bool need = false;
#pragma unroll
            for (int t = 0; t < TPS; ++t)
#pragma unroll
              for (int h = 0; h < NH; ++h) {
                if (!valid[t]) sc[t][h] = -INFINITY;
                need |= sc[t][h] > m_run[h] + 8.f;
              }
            // lazy rescaling: the reference max of a head moves only when a score of the step passes it by more
            // than 8 (a factor 2^8 in the weights)
            float alpha[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) alpha[h] = 1.f;
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
              for (int h = 0; h < NH; ++h) {
                float bm = sc[0][h];
#pragma unroll
                for (int t = 1; t < TPS; ++t) bm = fmaxf(bm, sc[t][h]);
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
                const float mn = fmaxf(m_run[h], bm);
                alpha[h] = ex2(m_run[h] - mn);
                m_run[h] = mn;
                l_run[h] *= alpha[h];
#pragma unroll
                for (int g = 0; g < NG; ++g) pb[g][h] *= alpha[h];
              }
            }
            float pr[TPS][NH];
#pragma unroll
            for (int t = 0; t < TPS; ++t)
#pragma unroll
              for (int h = 0; h < NH; ++h) {
                pr[t][h] = valid[t] ? ex2(sc[t][h] - m_run[h]) : 0.f;
                l_run[h] += pr[t][h];
              }
            // p * A_v for the V warps (buffer pbuf, free once the V warps are done with step j - 2), sums of p * B_v
            if (j >= 2) ok = ok && wait_warp(&p_empty[pbuf], ((j >> 1) - 1) & 1, abort_flag, p.err);
#pragma unroll
            for (int t = 0; t < TPS; ++t) {
              const int row = st * STEP + t * TILE + m;
              float4* psr = ps + ((size_t)pbuf * STEP + t * TILE + m) * Ls.ps_row;
              uint32_t vsw[NG / 2], vbw[NG / 2];
              load_halves<NG>(sVS + row * NG, vsw);
              load_halves<NG>(sVB + row * NG, vbw);
#pragma unroll
              for (int g = 0; g < NG; ++g) {
                const float sv =
                    valid[t] ? tc_half_to_float<DT>(half_of(vsw, g), f16) : 0.f;
                const float bv =
                    valid[t] ? tc_half_to_float<DT>(half_of(vbw, g), f16) : 0.f;
                const float2 av = tc_coeffs_v<FP32OUT>(sv, bv);
                if constexpr (PAIRED) {
                  const float2 p01 = __fmul2_rn(make_float2(pr[t][0], pr[t][1]), make_float2(av.x, av.x));
                  const float2 p23 = __fmul2_rn(make_float2(pr[t][2], pr[t][3]), make_float2(av.x, av.x));
                  psr[g] = make_float4(p01.x, p01.y, p23.x, p23.y);
                  const float2 b01 = __ffma2_rn(make_float2(pr[t][0], pr[t][1]), make_float2(av.y, av.y),
                                                make_float2(pb[g][0], pb[g][1]));
                  const float2 b23 = __ffma2_rn(make_float2(pr[t][2], pr[t][3]), make_float2(av.y, av.y),
                                                make_float2(pb[g][2], pb[g][3]));
                  pb[g][0] = b01.x;
                  pb[g][1] = b01.y;
                  pb[g][2] = b23.x;
                  pb[g][3] = b23.y;
                } else {
                  psr[g] = make_float4(pr[t][0] * av.x, pr[t][1] * av.x, pr[t][2] * av.x, pr[t][3] * av.x);
#pragma unroll
                  for (int h = 0; h < NH; ++h) pb[g][h] = fmaf(pr[t][h], av.y, pb[g][h]);
                }
              }
            }
            if (lane == 0)
              reinterpret_cast<float4*>(alpha_s)[pbuf * 4 + q] = make_float4(alpha[0], alpha[1], alpha[2], alpha[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[pbuf]);
          }
          if (c1 == walk.u_end || c1 == r1) {
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
              for (int h = 0; h < NH; ++h) {
                l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], off);
#pragma unroll
                for (int g = 0; g < NG; ++g) pb[g][h] += __shfl_xor_sync(0xffffffffu, pb[g][h], off);
              }
            }
            float* co = reinterpret_cast<float*>(vst);
            named_barrier_sync(1, EV_THREADS);   // the V warps are past this slot: it is free
            if (lane == 0) {
              float* cm = co + QDA_TC_VW * NH * D;
              float* cl = cm + 4 * NH;
              float* cpb = cl + 4 * NH;
#pragma unroll
              for (int h = 0; h < NH; ++h) {
                cm[q * NH + h] = m_run[h];
                cl[q * NH + h] = l_run[h];
#pragma unroll
                for (int g = 0; g < NG; ++g) cpb[(q * NG + g) * NH + h] = pb[g][h];
              }
            }
            combine(co, walk.unit);
            if (lane == 0) mbar_arrive(&qs_free[uidx & 1]);
            reset();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&vempty[vs]);
          ++i;
          if (++vs == VS) {
            vs = 0;
            vph ^= 1;
          }
        }
      } else {
        // ------------------------------------------------------------------------------ V warps
        const int vw = warp - V0;   // rows VROWS vw .. VROWS vw + VROWS - 1 of every step
        constexpr int VROWS = 16 * TPS;
        const int vlane = lane % VL, vrow = lane / VL;
        const int gv = (vlane * EV) / GS;
        float2 o[NH][EV / 2];
        auto reset = [&]() {
#pragma unroll
          for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int k = 0; k < EV / 2; ++k) o[h][k] = make_float2(0.f, 0.f);
        };
        reset();
        while (walk.next(p, c0, c1, t0)) {
          unsigned char* vst = smem + Ls.v0 + (size_t)vs * Ls.vstage_bytes;
          const int lr0 = (int)(c0 - t0), lr1 = (int)(c1 - t0);
          ok = ok && wait_warp(&vfull[vs], vph, abort_flag, p.err);
          const uint32_t* sV = reinterpret_cast<const uint32_t*>(vst);
          int st0, st1;
          tiles_of(lr0, lr1, st0, st1);
          for (int st = st0; st < st1; ++st, ++j) {
            const int pbuf = j & 1;
            ok = ok && wait_warp(&p_full[pbuf], (j >> 1) & 1, abort_flag, p.err);
            const float4 al4 = reinterpret_cast<const float4*>(alpha_s)[pbuf * 4 + q];
            const float al[4] = {al4.x, al4.y, al4.z, al4.w};
            if (al[0] != 1.f || al[1] != 1.f || al[2] != 1.f || al[3] != 1.f) {
#pragma unroll
              for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int k = 0; k < EV / 2; ++k) o[h][k] = __fmul2_rn(o[h][k], make_float2(al[h], al[h]));
            }
            const int rbase = st * STEP + VROWS * vw;   // this warp's slot rows (outside the chunk: p * A_v = 0)
            if (ok && rbase < lr1 && rbase + VROWS > lr0) {
              const float4* pp = ps + (size_t)pbuf * STEP * Ls.ps_row + gv;
#pragma unroll V_UNROLL
              for (int rs = 0; rs < VROWS / VR; ++rs) {
                const int r = VROWS * vw + rs * VR + vrow;   // step row
                uint32_t w[VW];
                load_words<VW>(sV + (st * STEP + r) * W + vlane * VW, w);
                float2 f[EV / 2];
                tc_unpack_v<FP32OUT, VW>(w, f);
                const float4 a4 = pp[r * Ls.ps_row];
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int h = 0; h < NH; ++h)
#pragma unroll
                  for (int k = 0; k < EV / 2; ++k) o[h][k] = __ffma2_rn(make_float2(av[h], av[h]), f[k], o[h][k]);
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_empty[pbuf]);
          }
          if (c1 == walk.u_end || c1 == r1) {
            if constexpr (VR > 1) {   // the lanes of one V slice took different rows: add their sums
#pragma unroll
              for (int off = VL; off < 32; off <<= 1)
#pragma unroll
                for (int h = 0; h < NH; ++h)
#pragma unroll
                  for (int k = 0; k < EV / 2; ++k)
                    o[h][k] = __fadd2_rn(o[h][k], make_float2(__shfl_xor_sync(0xffffffffu, o[h][k].x, off),
                                                              __shfl_xor_sync(0xffffffffu, o[h][k].y, off)));
            }
            float* co = reinterpret_cast<float*>(vst);
            named_barrier_sync(1, EV_THREADS);   // the epilogue warps are past this slot: it is free
            if (vrow == 0) {
#pragma unroll
              for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int k = 0; k < EV / 2; ++k)
                  reinterpret_cast<float2*>(co + ((2 * q + (TPS == 1 ? vw & 1 : vw >> 2)) * NH + h) * D +
                                            vlane * EV)[k] = o[h][k];
            }
            combine(co, walk.unit);
            reset();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&vempty[vs]);
          ++i;
          if (++vs == VS) {
            vs = 0;
            vph ^= 1;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// f16: q, scales and biases in fp16 (else bf16); the D = 128 instances take it as a template argument
template <bool FP32OUT, typename Fn>
cudaError_t with_tc_kernel(int D, int nh, int ng, bool f16, Fn&& f) {
#define QDA_TC(D_, NG_)                                                                          \
  if (D == D_ && nh == 4 && ng == NG_) {                                                         \
    if constexpr (D_ == 128)                                                                     \
      return f16 ? f(qda_tc_kernel<D_, 4, NG_, FP32OUT, 1>) : f(qda_tc_kernel<D_, 4, NG_, FP32OUT, 0>); \
    else                                                                                         \
      return f(qda_tc_kernel<D_, 4, NG_, FP32OUT, 2>);                                           \
  }
  QDA_TC(128, 2) QDA_TC(128, 4) QDA_TC(256, 2) QDA_TC(256, 4) QDA_TC(256, 8)
#undef QDA_TC
  return cudaErrorInvalidValue;
}

}  // namespace qda
