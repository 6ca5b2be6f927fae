// Affine-quantized weight GEMV (sm_103a), the comparison workload for the cache codec:
//     y[t, n] = sum_k x[t, k] * (scale[n, k / GS] * code[n, k] + bias[n, k / GS]),   t < T <= 4
// (maya-mac mlx_kernels.py, _linear_kernel with 8-bit weights: one simdgroup per group of output rows, lanes
// striding along K, dequantisation inlined; its LayerNorm, activation and residual epilogues are model-specific and
// not part of this workload).
//
// S warps own R = 4 output rows, each taking 1/S of K (S = 1, 2 or 4, chosen so that a wide matrix still spreads
// over every SM); each step a lane takes 128 bits of codes (16 elements of 8-bit, 32 of 4-bit) per row, copied
// past L1 into its own slots of a shared-memory ring two steps ahead (asynchronous 16-byte copies: the loads in
// flight hold no registers), the x slice of those elements (read through the read-only path: every warp reads the same few KB of x),
// and the row's scale and bias of that group. The dot is factored as in the attention kernels: s * sum(x * code) +
// b * sum(x), with exact codes (a byte permute to 2^23 + code, minus 2^23) and packed f32x2 FMAs. Lanes reduce
// by shuffles, the S parts meet in shared memory in a fixed order, and one lane writes the rounded outputs. The
// weights are streamed once: a matrix-vector product is bound by HBM.
#include <algorithm>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qda_internal.h"
#include "qda_ptx.cuh"

namespace qda {

constexpr int kGemvThreads = 256;
constexpr int kGemvRows = 4;      // output rows per warp
constexpr int kGemvWarps = kGemvThreads / 32;
// depth of each lane's shared-memory ring of code loads: STAGES - 1 steps are in flight while one is worked on
// (measured at K = 4096, N = 14336: 3 stages 8 % faster than one step ahead in registers for one input row of
// 8-bit codes and 9 % for two rows of 4-bit codes; 4 and 6 stages no faster)
constexpr int kGemvStages = 3;
// dynamic shared memory of one CTA: per warp STAGES steps of R rows x 32 lanes x 16 bytes
constexpr size_t kGemvRingBytes = (size_t)kGemvWarps * kGemvStages * kGemvRows * 32 * 16;

// 16-byte asynchronous copy global -> shared (L2 only), and its group commit / wait; a thread waits for its own copies
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// elements of K per lane per step: one 128-bit load of codes
template <int BITS>
__host__ __device__ constexpr int gemv_codes() { return 128 / BITS; }

// The codes of one word as exact float pairs (code 2j, code 2j + 1): a byte permute puts each code under the
// exponent byte of 2^23 ([code, 0, 0, 0x4B] = 2^23 + code) and one packed subtract removes 2^23.
template <int BITS>
__device__ __forceinline__ void word_to_float(uint32_t w, float2 (&c)[16 / BITS]) {
  const float2 off = make_float2(-8388608.0f, -8388608.0f);
  if constexpr (BITS == 8) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      c[j] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u | (2 * j))),
                                    __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7651u | (2 * j)))), off);
  } else {
    const uint32_t lo = w & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6 of the word in bytes 0..3
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
#pragma unroll
    for (int j = 0; j < 4; ++j)
      c[j] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7650u | j)),
                                    __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7650u | j))), off);
  }
}

template <int OUT>
__device__ __forceinline__ void store_out(void* y, size_t idx, float v) {
  if constexpr (OUT == QDA_FP32) {
    static_cast<float*>(y)[idx] = v;
  } else if constexpr (OUT == QDA_BF16) {
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(y)[idx] = __float2half_rn(v);
  }
}

// resident CTAs per SM the register budget aims at: three for one input row of 8-bit codes, fewer as the x slice
// (4-bit codes: 32 elements a step) and the accumulators grow; F16: x, scales and biases in fp16 (else bf16), a
// template argument so that each conversion is one instruction
template <int BITS, int T, int OUT, bool F16>
__global__ void __launch_bounds__(kGemvThreads, T == 1 ? (BITS == 8 ? 3 : 2) : (T == 2 && BITS == 8) ? 2 : 1)
    qda_qgemv_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ wp, const uint16_t* __restrict__ ws,
                     const uint16_t* __restrict__ wb, void* __restrict__ y, int N, int K, int GS, int S) {
  constexpr int R = kGemvRows, C = gemv_codes<BITS>(), ST = kGemvStages;
  __shared__ float part[kGemvWarps][R][T];
  extern __shared__ uint4 gemv_ring[];   // [warp][stage][row][lane]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / S, sp = warp - grp * S;       // row group within the CTA's block of rows, K part
  const int kpart = K / S, kbeg = sp * kpart;
  const int W = K * BITS / 32, NG = K / GS;
  const int rows_per_block = (kGemvWarps / S) * R;
  const int blocks = (N + rows_per_block - 1) / rows_per_block;
  // a grid of whole waves (SMs x resident CTAs) takes the blocks of rows in turn
  for (int blk = blockIdx.x; blk < blocks; blk += gridDim.x) {
    const int n0 = blk * rows_per_block + grp * R;
    float2 acc[R][T];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < T; ++t) acc[r][t] = make_float2(0.f, 0.f);
    float bacc[R][T];   // sum of bias * sum(x) per row and input
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < T; ++t) bacc[r][t] = 0.f;

    // the codes of the R rows go through a ring of ST steps in shared memory, filled by asynchronous copies ST - 1
    // steps ahead: each lane copies its own 16 bytes per row and step and reads back only those, so its own group
    // waits order them and no other lane is involved
    const bool live = n0 < N;
    const int nsteps = kpart / (32 * C);
    uint4* ring = gemv_ring + (size_t)warp * ST * R * 32 + lane;
    auto issue = [&](int step) {
      if (live && step < nsteps) {
        const int ks = kbeg + step * 32 * C + lane * C;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int n = min(n0 + r, N - 1);   // rows past N repeat the last row; their results are not written
          cp_async16(ring + ((step % ST) * R + r) * 32, wp + (size_t)n * W + (size_t)ks * BITS / 32);
        }
      }
      cp_async_commit();   // an empty group past the end keeps the count of pending groups in step
    };
#pragma unroll
    for (int st = 0; st < ST - 1; ++st) issue(st);
    for (int step = 0; live && step < nsteps; ++step) {
      issue(step + ST - 1);   // into the slot read one step ago: its values are in registers and used
      cp_async_wait<ST - 1>();
      const int k0 = kbeg + step * 32 * C + lane * C;
      uint4 cur[R];
#pragma unroll
      for (int r = 0; r < R; ++r) cur[r] = ring[((step % ST) * R + r) * 32];
      // the x slice of these C elements, and its sums
      float2 xv[T][C / 2];
      float xs[T];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)t * K + k0);
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < C / 8; ++q) {
          const uint4 a = __ldg(xp + q);
          const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            xv[t][4 * q + i] = make_float2(half_bits_to_float<F16>(u[i] & 0xFFFFu), half_bits_to_float<F16>(u[i] >> 16));
            sum += xv[t][4 * q + i].x + xv[t][4 * q + i].y;
          }
        }
        xs[t] = sum;
      }
      const int g = k0 / GS;   // a lane's C elements lie in one group (C <= GS)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int n = min(n0 + r, N - 1);
        const float s = half_bits_to_float<F16>(__ldg(ws + (size_t)n * NG + g));
        const float b = half_bits_to_float<F16>(__ldg(wb + (size_t)n * NG + g));
        // one word of codes at a time: only its pairs are live
        constexpr int PW = 16 / BITS;   // code pairs per word
        const uint32_t wv[4] = {cur[r].x, cur[r].y, cur[r].z, cur[r].w};
        float2 d[T];
#pragma unroll
        for (int t = 0; t < T; ++t) d[t] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 c[PW];
          word_to_float<BITS>(wv[i], c);
#pragma unroll
          for (int t = 0; t < T; ++t)
#pragma unroll
            for (int j = 0; j < PW; ++j) d[t] = __ffma2_rn(c[j], xv[t][PW * i + j], d[t]);
        }
#pragma unroll
        for (int t = 0; t < T; ++t) {
          acc[r][t] = __ffma2_rn(make_float2(s, s), d[t], acc[r][t]);
          bacc[r][t] = fmaf(b, xs[t], bacc[r][t]);
        }
      }
    }
    cp_async_wait<0>();   // nothing of this block in flight when the ring is refilled for the next
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float v = acc[r][t].x + acc[r][t].y + bacc[r][t];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (S == 1) {   // one part: the warp writes its rows itself
          if (lane == 0 && n0 + r < N) store_out<OUT>(y, (size_t)t * N + n0 + r, v);
        } else if (lane == 0) {
          part[warp][r][t] = v;
        }
      }
    if (S > 1) {
      __syncthreads();
      if (sp == 0 && lane < R * T) {   // the S parts of this row group, added in order
        const int r = lane / T, t = lane - r * T;
        float v = 0.f;
        for (int q = 0; q < S; ++q) v += part[warp + q][r][t];
        if (n0 + r < N) store_out<OUT>(y, (size_t)t * N + n0 + r, v);
      }
      __syncthreads();   // the partials are read before the next block of rows overwrites them
    }
  }
}

template <int BITS, int T>
cudaError_t launch_qgemv_t(const uint16_t* x, const uint32_t* wp, const uint16_t* ws, const uint16_t* wb, void* y,
                           int N, int K, int GS, int f16, int out, int sms, cudaStream_t s) {
  // K parts per row group: the fewest that give every SM four blocks of rows, as K allows (whole 32-lane steps)
  int S = 1;
  while (S < 4 && (long long)(N + (kGemvWarps / S) * kGemvRows - 1) / ((kGemvWarps / S) * kGemvRows) < 4LL * sms &&
         K % (32 * gemv_codes<BITS>() * S * 2) == 0)
    S *= 2;
  const int rows_per_cta = (kGemvWarps / S) * kGemvRows;
  const long long blocks = (N + rows_per_cta - 1) / rows_per_cta;
  auto pick = [&](auto f16) {
    constexpr bool F = decltype(f16)::value;
    return out == QDA_BF16 ? qda_qgemv_kernel<BITS, T, QDA_BF16, F>
         : out == QDA_FP16 ? qda_qgemv_kernel<BITS, T, QDA_FP16, F> : qda_qgemv_kernel<BITS, T, QDA_FP32, F>;
  };
  auto kern = f16 ? pick(std::true_type{}) : pick(std::false_type{});
  static int occ[3][2] = {};   // resident CTAs per SM of each instance (the same on every GB300)
  int& o = occ[out == QDA_BF16 ? 0 : out == QDA_FP16 ? 1 : 2][f16 ? 1 : 0];
  if (o == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvRingBytes);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kGemvThreads, kGemvRingBytes);
    if (e != cudaSuccess) return e;
    if (o < 1) o = 1;
  }
  const dim3 grid((unsigned)std::min<long long>(blocks, (long long)sms * o));
  kern<<<grid, kGemvThreads, kGemvRingBytes, s>>>(x, wp, ws, wb, y, N, K, GS, S);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_qgemv(const uint16_t* x, const uint32_t* wp, const uint16_t* ws, const uint16_t* wb, void* y,
                         int T, int N, int K, int GS, int f16, int out, int sms, cudaStream_t s) {
  switch (T) {
    case 1: return launch_qgemv_t<BITS, 1>(x, wp, ws, wb, y, N, K, GS, f16, out, sms, s);
    case 2: return launch_qgemv_t<BITS, 2>(x, wp, ws, wb, y, N, K, GS, f16, out, sms, s);
    case 3: return launch_qgemv_t<BITS, 3>(x, wp, ws, wb, y, N, K, GS, f16, out, sms, s);
    default: return launch_qgemv_t<BITS, 4>(x, wp, ws, wb, y, N, K, GS, f16, out, sms, s);
  }
}

}  // namespace qda

extern "C" int qdecode_qgemv(const void* x, const uint32_t* w_packed, const void* w_scales, const void* w_biases,
                             void* y, int T, int N, int K, int GS, int bits, int dtype, void* stream) {
  if (!x || !w_packed || !w_scales || !w_biases || !y) return QDA_ERR_INVALID;
  if (T < 1 || N < 1 || K < 1 || GS < 1) return QDA_ERR_INVALID;
  const int in_dt = dtype & 0xff, out_byte = (dtype >> 8) & 0xff;
  if ((dtype >> 16) != 0 || (in_dt != QDA_BF16 && in_dt != QDA_FP16)) return QDA_ERR_INVALID;
  if (out_byte != 0 && out_byte != QDA_BF16 && out_byte != QDA_FP16 && out_byte != QDA_FP32) return QDA_ERR_INVALID;
  const int out_dt = out_byte == 0 ? in_dt : out_byte;
  if (bits != 4 && bits != 8) return QDA_ERR_UNSUPPORTED;
  if (GS != 32 && GS != 64 && GS != 128) return QDA_ERR_UNSUPPORTED;
  if (T > QDA_QGEMV_MAX_T || K % (32 * 128 / bits) != 0) return QDA_ERR_UNSUPPORTED;   // whole 32-lane steps
  const void* ptrs[5] = {x, w_packed, w_scales, w_biases, y};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return QDA_ERR_ALIGN;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  const uint16_t* ws = static_cast<const uint16_t*>(w_scales);
  const uint16_t* wb = static_cast<const uint16_t*>(w_biases);
  const int f16 = in_dt == QDA_FP16;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return qda_cuda_fail(e);
  e = bits == 8 ? qda::launch_qgemv<8>(xs, w_packed, ws, wb, y, T, N, K, GS, f16, out_dt, sms, s)
                : qda::launch_qgemv<4>(xs, w_packed, ws, wb, y, T, N, K, GS, f16, out_dt, sms, s);
  if (e != cudaSuccess) return qda_cuda_fail(e);
  return QDA_OK;
}
