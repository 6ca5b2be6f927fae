// Affine-quantized weight GEMV (sm_103a), the comparison workload for the cache codec:
//     y[t, n] = sum_k x[t, k] * (scale[n, k / GS] * code[n, k] + bias[n, k / GS]),   t < T <= 4
// (maya-mac mlx_kernels.py, _linear_kernel with 8-bit weights: one simdgroup per group of output rows, lanes
// striding along K, dequantisation inlined; its LayerNorm, activation and residual epilogues are model-specific and
// not part of this workload).
//
// One warp owns R = 4 output rows; each step a lane takes 16 consecutive elements of K (one 16- or 8-byte load
// per row, streamed past L1), the x slice of those elements (read through the read-only path: every warp of the
// GPU reads the same few KB of x), and the row's scale and bias of that group. The dot is factored as in the
// attention kernels: s * sum(x * code) + b * sum(x), with exact codes (2^23 + code minus 2^23) and packed f32x2
// FMAs. Lanes then reduce by shuffles and lane 0 writes the rounded outputs. A warp-per-row-group GEMV streams the
// weights once with no shared memory, which is all a matrix-vector product needs: it is bound by HBM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qda_internal.h"
#include "qda_ptx.cuh"

namespace qda {

constexpr int kGemvThreads = 256;
constexpr int kGemvRows = 4;      // output rows per warp
constexpr int kGemvCodes = 16;    // elements of K per lane per step

template <int BITS>
__device__ __forceinline__ void load_codes(const uint32_t* p, uint32_t (&w)[kGemvCodes * BITS / 32]) {
  if constexpr (BITS == 8) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
    w[0] = v.x;
    w[1] = v.y;
  }
}

// codes of the words as exact floats, in element order
template <int BITS>
__device__ __forceinline__ void codes_to_float(const uint32_t (&w)[kGemvCodes * BITS / 32], float (&c)[kGemvCodes]) {
  constexpr int PER = 32 / BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
#pragma unroll
  for (int i = 0; i < kGemvCodes * BITS / 32; ++i)
#pragma unroll
    for (int k = 0; k < PER; ++k)
      c[i * PER + k] = __uint_as_float(0x4B000000u | ((w[i] >> (BITS * k)) & MASK)) - 8388608.0f;
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

template <int BITS, int T, int OUT>
__global__ void __launch_bounds__(kGemvThreads) qda_qgemv_kernel(const uint16_t* __restrict__ x,
                                                                const uint32_t* __restrict__ wp,
                                                                const uint16_t* __restrict__ ws,
                                                                const uint16_t* __restrict__ wb, void* __restrict__ y,
                                                                int N, int K, int GS, int f16) {
  constexpr int R = kGemvRows, C = kGemvCodes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = (blockIdx.x * (kGemvThreads / 32) + warp) * R;
  if (n0 >= N) return;
  const int W = K * BITS / 32, NG = K / GS;
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

  for (int k0 = lane * C; k0 < K; k0 += 32 * C) {
    // the x slice of these 16 elements, and its sums
    float2 xv[T][C / 2];
    float xs[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)t * K + k0);
      const uint4 a = __ldg(xp), b = __ldg(xp + 1);
      const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xv[t][i] = make_float2(half_bits_to_float_rt(u[i] & 0xFFFFu, f16 != 0),
                               half_bits_to_float_rt(u[i] >> 16, f16 != 0));
        sum += xv[t][i].x + xv[t][i].y;
      }
      xs[t] = sum;
    }
    const int g = k0 / GS;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int n = min(n0 + r, N - 1);   // rows past N repeat the last row; their results are not written
      uint32_t w[C * BITS / 32];
      load_codes<BITS>(wp + (size_t)n * W + (size_t)k0 * BITS / 32, w);
      const float s = half_bits_to_float_rt(__ldg(ws + (size_t)n * NG + g), f16 != 0);
      const float b = half_bits_to_float_rt(__ldg(wb + (size_t)n * NG + g), f16 != 0);
      float c[C];
      codes_to_float<BITS>(w, c);
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float2 d = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < C / 2; ++i) d = __ffma2_rn(make_float2(c[2 * i], c[2 * i + 1]), xv[t][i], d);
        acc[r][t] = __ffma2_rn(make_float2(s, s), d, acc[r][t]);
        bacc[r][t] = fmaf(b, xs[t], bacc[r][t]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float v = acc[r][t].x + acc[r][t].y + bacc[r][t];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && n0 + r < N) store_out<OUT>(y, (size_t)t * N + n0 + r, v);
    }
}

template <int BITS, int T>
cudaError_t launch_qgemv_t(const uint16_t* x, const uint32_t* wp, const uint16_t* ws, const uint16_t* wb, void* y,
                           int N, int K, int GS, int f16, int out, cudaStream_t s) {
  const int rows_per_cta = (kGemvThreads / 32) * kGemvRows;
  const dim3 grid((unsigned)((N + rows_per_cta - 1) / rows_per_cta));
  switch (out) {
    case QDA_BF16: qda_qgemv_kernel<BITS, T, QDA_BF16><<<grid, kGemvThreads, 0, s>>>(x, wp, ws, wb, y, N, K, GS, f16); break;
    case QDA_FP16: qda_qgemv_kernel<BITS, T, QDA_FP16><<<grid, kGemvThreads, 0, s>>>(x, wp, ws, wb, y, N, K, GS, f16); break;
    default: qda_qgemv_kernel<BITS, T, QDA_FP32><<<grid, kGemvThreads, 0, s>>>(x, wp, ws, wb, y, N, K, GS, f16); break;
  }
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_qgemv(const uint16_t* x, const uint32_t* wp, const uint16_t* ws, const uint16_t* wb, void* y,
                         int T, int N, int K, int GS, int f16, int out, cudaStream_t s) {
  switch (T) {
    case 1: return launch_qgemv_t<BITS, 1>(x, wp, ws, wb, y, N, K, GS, f16, out, s);
    case 2: return launch_qgemv_t<BITS, 2>(x, wp, ws, wb, y, N, K, GS, f16, out, s);
    case 3: return launch_qgemv_t<BITS, 3>(x, wp, ws, wb, y, N, K, GS, f16, out, s);
    default: return launch_qgemv_t<BITS, 4>(x, wp, ws, wb, y, N, K, GS, f16, out, s);
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
  if (T > QDA_QGEMV_MAX_T || K % 512 != 0) return QDA_ERR_UNSUPPORTED;
  const void* ptrs[5] = {x, w_packed, w_scales, w_biases, y};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return QDA_ERR_ALIGN;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  const uint16_t* ws = static_cast<const uint16_t*>(w_scales);
  const uint16_t* wb = static_cast<const uint16_t*>(w_biases);
  const int f16 = in_dt == QDA_FP16;
  const cudaError_t e = bits == 8 ? qda::launch_qgemv<8>(xs, w_packed, ws, wb, y, T, N, K, GS, f16, out_dt, s)
                                  : qda::launch_qgemv<4>(xs, w_packed, ws, wb, y, T, N, K, GS, f16, out_dt, s);
  if (e != cudaSuccess) return qda_cuda_fail(e);
  return QDA_OK;
}
