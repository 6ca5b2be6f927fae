// Merge kernel (fixed-order combine of the split partials), the cache quantizer and the cache-append copy, sm_103a.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qda_internal.h"
#include "qda_ptx.cuh"

namespace qda {

__device__ __forceinline__ float ex2m(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int OUT>
__device__ __forceinline__ void store4(void* out, size_t idx, float4 v) {
  if constexpr (OUT == QDA_FP32) {
    reinterpret_cast<float4*>(out)[idx] = v;
  } else if constexpr (OUT == QDA_BF16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[idx] = u;
  } else {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[idx] = u;
  }
}

// out[b, l, h, :] = sum_s o_s 2^(m_s - M) / sum_s l_s 2^(m_s - M) over the partial slots of (b, KV head of h)
// (mlx-bun fused-decode-kernel.ts, MERGE_SOURCE), in log2 units. One CTA per (b, l, h) and slice of the head
// dimension (gridDim.y slices; one, or 64 values each when a head has many slots); l is the query position
// (always 0 for single-query decode). A slot whose rows were all hidden
// from the head holds m = -inf and is skipped. In compat mode (the two-pass form) the partials already carry
// normalised weights and are only summed (in the same fixed order): out = T(sum_s o_s). The slots are dealt to
// THREADS / (slice / 4) thread groups round-robin (4 values per thread); each thread folds its slots
// in one pass with a running max, so the (m, l) and o loads of a slot are issued together, and the groups are then
// combined in a fixed order: deterministic, no atomics.
// Threads per merge CTA: 512, or 1024 when the merge has few CTAs (one per head and slice, at most an eighth of the
// SMs): the SMs are idle then, and each thread folds half as many slots (8k workload: the call 0.35 us shorter; with
// many CTAs the larger blocks were 1-4 us slower).
constexpr int kMergeThreads = 512;

template <int OUT, int THREADS>
__global__ void __launch_bounds__(THREADS) qda_merge_kernel(const __grid_constant__ QdaParams p,
                                                            void* __restrict__ out) {
  __shared__ float4 red_o[THREADS];
  __shared__ float2 red_ml[THREADS];
  const int tid = threadIdx.x;
  const int D = p.D;
  const int bh = blockIdx.x;   // (b * L + l) * H + h: also the output row
  const int bl = bh / p.H, h = bh - bl * p.H;
  const int b = bl / p.L, l = bl - b * p.L;
  const int kvh = h / p.nrep, j = l * p.nrep + (h - kvh * p.nrep);
  const int unit = b * p.Hkv + kvh;
  const long long n = p.seq_off[b + 1] - p.seq_off[b];
  const long long us = (long long)p.Hkv * p.seq_off[b] + (long long)kvh * n;
  const long long T = p.total_rows;
  const int C = p.num_ctas;
  const int cf = qda_cta_of(T, C, us);
  const int ns = qda_cta_of(T, C, us + n - 1) - cf + 1;
  const bool maybe_empty = T / C < 8;   // only ranges shorter than 8 rows can be empty (and wrote no slot)
  // this CTA's slice of the head dimension (gridDim.y slices of D / gridDim.y values), 4 values per thread
  const int dims = D / (int)gridDim.y;
  const int tpr = dims >> 2;
  const int groups = THREADS / tpr;
  const int grp = tid / tpr, t = (int)blockIdx.y * tpr + (tid - grp * tpr);

  pdl_launch_dependents();   // the next call's split kernel may launch now (it waits for this grid before any access)
  pdl_wait();   // the split kernel's partials are complete and visible from here on

  float m_run = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int k = grp; k < ns; k += groups) {
    const int c = cf + k;
    if (!in_bounds(c + unit < C + p.B * p.Hkv && j < p.heads_pad, p.err)) continue;
    const size_t hp = (size_t)(c + unit) * p.heads_pad + j;
    const float2 ml = p.part_ml[hp];
    const float4 v = reinterpret_cast<const float4*>(p.part_o + hp * D)[t];
    if (maybe_empty && qda_cta_row(T, C, c) == qda_cta_row(T, C, c + 1)) continue;
    // a slot whose rows were all hidden from this query position holds (m, l, o) = (-inf, 0, 0): taken as a
    // finite m it adds nothing and never forms -inf - -inf
    const float mx = p.compat ? 0.f : fmaxf(ml.x, -1e30f);   // compat: every slot weighs 1
    const float mn = fmaxf(m_run, mx);
    const float a = ex2m(m_run - mn);   // 0 on the first slot
    const float w = ex2m(mx - mn);
    den = fmaf(den, a, (p.compat ? 0.f : ml.y) * w);
    acc.x = fmaf(acc.x, a, v.x * w);
    acc.y = fmaf(acc.y, a, v.y * w);
    acc.z = fmaf(acc.z, a, v.z * w);
    acc.w = fmaf(acc.w, a, v.w * w);
    m_run = mn;
  }
  red_o[tid] = acc;
  if (tid - grp * tpr == 0) red_ml[grp] = make_float2(m_run, den);
  __syncthreads();
  if (grp != 0) return;
  float M = -INFINITY;
  for (int g = 0; g < groups; ++g) M = fmaxf(M, red_ml[g].x);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float dt = 0.f;
  for (int g = 0; g < groups; ++g) {
    const float2 ml = red_ml[g];
    if (ml.x == -INFINITY) continue;   // a group that held no slot
    const float w = ex2m(ml.x - M);
    const float4 v = red_o[g * tpr + tid];
    dt = fmaf(ml.y, w, dt);
    o.x = fmaf(v.x, w, o.x);
    o.y = fmaf(v.y, w, o.y);
    o.z = fmaf(v.z, w, o.z);
    o.w = fmaf(v.w, w, o.w);
  }
  const float inv = p.compat ? 1.f : 1.0f / dt;
  o.x *= inv;
  o.y *= inv;
  o.z *= inv;
  o.w *= inv;
  store4<OUT>(out, ((size_t)bh * D >> 2) + t, o);
}

// ------------------------------------------------------------------------------------------- quantizer

template <bool F16>
__device__ __forceinline__ uint32_t round_bits16(float x) {
  if constexpr (F16) {
    return __half_as_ushort(__float2half_rn(x));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
}

// One warp per row of D = 32 * E fp32 values; lane l holds elements [l*E, l*E + E). A group spans GS/E lanes.
__device__ __forceinline__ long long mapped_row(const QdaRowMap& m, long long i) {
  if (!m.append) return i;
  const int per_seq = m.Hkv * m.T;
  const int b = (int)(i / per_seq);
  const int rem = (int)(i - (long long)b * per_seq);
  const int kvh = rem / m.T, t = rem - kvh * m.T;
  return (long long)m.Hkv * m.off_new[b] + (long long)kvh * (m.n_old[b] + m.T) + m.n_old[b] + t;
}

template <int BITS, int E, bool F16>
__global__ void __launch_bounds__(256) qda_quant_kernel(const float* __restrict__ x, long long rows, int GS,
                                                        uint32_t* __restrict__ packed, uint16_t* __restrict__ sc,
                                                        uint16_t* __restrict__ bi, const __grid_constant__ QdaRowMap map) {
  constexpr int D = 32 * E;
  constexpr int PER = 32 / BITS;
  constexpr int W = D / PER;
  constexpr float QMAX = (float)((1 << BITS) - 1);
  // launched behind another kernel of the same cache append (programmatic dependent launch), this one may start
  // early: it reads nothing the other writes. It finishes only after its predecessor has (griddepcontrol.wait at
  // the end, a no-op for an ordinary launch), so the append's last kernel completing means the whole append is done.
  pdl_launch_dependents();
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) {
    pdl_wait();
    return;
  }
  const int lane = threadIdx.x & 31;
  const float* xr = x + row * D + lane * E;
  const long long orow = mapped_row(map, row);   // the row written
  float v[E];
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int k = 0; k < E / 4; ++k) {
      const float4 t = reinterpret_cast<const float4*>(xr)[k];
      v[4 * k] = t.x;
      v[4 * k + 1] = t.y;
      v[4 * k + 2] = t.z;
      v[4 * k + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
      const float2 t = reinterpret_cast<const float2*>(xr)[k];
      v[2 * k] = t.x;
      v[2 * k + 1] = t.y;
    }
  }
  float lo = v[0], hi = v[0];
#pragma unroll
  for (int e = 1; e < E; ++e) {
    lo = fminf(lo, v[e]);
    hi = fmaxf(hi, v[e]);
  }
  const int lpg = GS / E;
  for (int off = 1; off < lpg; off <<= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
  }
  const float scale = __fdiv_rn(__fsub_rn(hi, lo), QMAX);
  const uint32_t sbits = round_bits16<F16>(scale);
  const uint32_t bbits = round_bits16<F16>(lo);
  const float s_hat = half_bits_to_float<F16>(sbits);
  const float b_hat = half_bits_to_float<F16>(bbits);
  uint32_t code[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float r = rintf(__fdiv_rn(__fsub_rn(v[e], b_hat), s_hat));
    r = fminf(fmaxf(r, 0.f), QMAX);
    code[e] = (s_hat == 0.f) ? 0u : (uint32_t)r;
  }
  if constexpr (E * BITS >= 32) {
    constexpr int WL = E * BITS / 32;  // whole words per lane
#pragma unroll
    for (int w = 0; w < WL; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < PER; ++k) word |= code[w * PER + k] << (BITS * k);
      packed[orow * W + lane * WL + w] = word;
    }
  } else {
    constexpr int LPW = 32 / (E * BITS);  // lanes sharing a word
    uint32_t part = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) part |= code[e] << (BITS * e);
    part <<= (E * BITS) * (lane % LPW);
#pragma unroll
    for (int off = 1; off < LPW; off <<= 1) part |= __shfl_xor_sync(0xffffffffu, part, off);
    if (lane % LPW == 0) packed[orow * W + lane / LPW] = part;
  }
  if ((lane * E) % GS == 0) {
    const int NG = D / GS;
    sc[orow * NG + (lane * E) / GS] = (uint16_t)sbits;
    bi[orow * NG + (lane * E) / GS] = (uint16_t)bbits;
  }
  pdl_wait();
}

// Copies the old rows of the (sequence, KV head) units into the appended cache: CTA (x, y) takes rows
// [x * kAppendRows, (x + 1) * kAppendRows) of units y, y + gridDim.y, ... A unit's old rows are contiguous in both caches (its block
// only moves by the new rows of the blocks before it), so the K and V codes go as flat 16-byte pieces and the
// scales and biases as flat pairs of 16-bit values (NG is even); streaming loads and stores, four 16-byte pieces of K
// and of V in flight per thread. Launched behind the append's quantizer launches with programmatic dependent launch
// (see qda_quant_kernel).
constexpr int kAppendRows = 128;

__global__ void __launch_bounds__(256) qda_append_copy_kernel(
    const uint32_t* __restrict__ kp, const uint16_t* __restrict__ ks, const uint16_t* __restrict__ kb,
    const uint32_t* __restrict__ vp, const uint16_t* __restrict__ vs, const uint16_t* __restrict__ vb,
    uint32_t* __restrict__ kpo, uint16_t* __restrict__ kso, uint16_t* __restrict__ kbo, uint32_t* __restrict__ vpo,
    uint16_t* __restrict__ vso, uint16_t* __restrict__ vbo, int W, int NG, const __grid_constant__ QdaRowMap m) {
  for (int unit = blockIdx.y; unit < m.B * m.Hkv; unit += gridDim.y) {
    const int b = unit / m.Hkv, kvh = unit - b * m.Hkv;
    const long long n = m.n_old[b];
    const long long r0 = (long long)blockIdx.x * kAppendRows;
    if (r0 >= n) continue;
    const long long rows = min((long long)kAppendRows, n - r0);
    const long long src = (long long)m.Hkv * m.off_old[b] + kvh * n + r0;              // first row, old cache
    const long long dst = (long long)m.Hkv * m.off_new[b] + kvh * (n + m.T) + r0;      // its row, new cache
    const int cpr = W / 4;   // 16-byte pieces per row
    const uint4* k4 = reinterpret_cast<const uint4*>(kp) + src * cpr;
    const uint4* v4 = reinterpret_cast<const uint4*>(vp) + src * cpr;
    uint4* ko4 = reinterpret_cast<uint4*>(kpo) + dst * cpr;
    uint4* vo4 = reinterpret_cast<uint4*>(vpo) + dst * cpr;
    const long long pieces = rows * cpr;
    const long long step = blockDim.x;
    long long i = threadIdx.x;
    for (; i + 3 * step < pieces; i += 4 * step) {
      uint4 a[4], c[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = __ldcs(k4 + i + u * step);
        c[u] = __ldcs(v4 + i + u * step);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        __stcs(ko4 + i + u * step, a[u]);
        __stcs(vo4 + i + u * step, c[u]);
      }
    }
    for (; i < pieces; i += step) {
      const uint4 a = __ldcs(k4 + i), c = __ldcs(v4 + i);
      __stcs(ko4 + i, a);
      __stcs(vo4 + i, c);
    }
    // a row's NG 16-bit values start at a multiple of 2 * NG bytes: 32-bit pairs
    const long long e = rows * NG / 2;
    const uint32_t *ks2 = reinterpret_cast<const uint32_t*>(ks + src * NG), *kb2 = reinterpret_cast<const uint32_t*>(kb + src * NG);
    const uint32_t *vs2 = reinterpret_cast<const uint32_t*>(vs + src * NG), *vb2 = reinterpret_cast<const uint32_t*>(vb + src * NG);
    uint32_t *kso2 = reinterpret_cast<uint32_t*>(kso + dst * NG), *kbo2 = reinterpret_cast<uint32_t*>(kbo + dst * NG);
    uint32_t *vso2 = reinterpret_cast<uint32_t*>(vso + dst * NG), *vbo2 = reinterpret_cast<uint32_t*>(vbo + dst * NG);
    for (long long k = threadIdx.x; k < e; k += step) {
      const uint32_t x0 = ks2[k], x1 = kb2[k], x2 = vs2[k], x3 = vb2[k];
      kso2[k] = x0;
      kbo2[k] = x1;
      vso2[k] = x2;
      vbo2[k] = x3;
    }
  }
  pdl_wait();
}

template <int BITS, bool F16>
cudaError_t launch_quant(const float* x, long long rows, int D, int GS, uint32_t* packed, uint16_t* sc, uint16_t* bi,
                         cudaStream_t s, const QdaRowMap& m, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (D) {
    case 64: return cudaLaunchKernelEx(&cfg, qda_quant_kernel<BITS, 2, F16>, x, rows, GS, packed, sc, bi, m);
    case 128: return cudaLaunchKernelEx(&cfg, qda_quant_kernel<BITS, 4, F16>, x, rows, GS, packed, sc, bi, m);
    case 256: return cudaLaunchKernelEx(&cfg, qda_quant_kernel<BITS, 8, F16>, x, rows, GS, packed, sc, bi, m);
    case 512: return cudaLaunchKernelEx(&cfg, qda_quant_kernel<BITS, 16, F16>, x, rows, GS, packed, sc, bi, m);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qda

cudaError_t qda_launch_merge(const QdaParams& p, void* out, int out_dtype, bool pdl, int slices, int num_sms,
                             cudaStream_t s) {
  if (slices < 1 || p.D % (4 * slices) != 0 || p.D / 4 / slices > qda::kMergeThreads) return cudaErrorInvalidValue;
  const long long ctas = (long long)p.B * p.L * p.H * slices;
  const bool wide = ctas * 8 <= num_sms;   // few merge CTAs: 1024 threads each
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.L * p.H), (unsigned)slices);
  cfg.blockDim = dim3(wide ? 2 * qda::kMergeThreads : qda::kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  constexpr int T1 = qda::kMergeThreads, T2 = 2 * qda::kMergeThreads;
  switch (out_dtype) {
    case QDA_BF16:
      return wide ? cudaLaunchKernelEx(&cfg, qda::qda_merge_kernel<QDA_BF16, T2>, p, out)
                  : cudaLaunchKernelEx(&cfg, qda::qda_merge_kernel<QDA_BF16, T1>, p, out);
    case QDA_FP16:
      return wide ? cudaLaunchKernelEx(&cfg, qda::qda_merge_kernel<QDA_FP16, T2>, p, out)
                  : cudaLaunchKernelEx(&cfg, qda::qda_merge_kernel<QDA_FP16, T1>, p, out);
    case QDA_FP32:
      return wide ? cudaLaunchKernelEx(&cfg, qda::qda_merge_kernel<QDA_FP32, T2>, p, out)
                  : cudaLaunchKernelEx(&cfg, qda::qda_merge_kernel<QDA_FP32, T1>, p, out);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t qda_launch_quantize(const float* x, long long rows, int D, int GS, int bits, int in_dtype,
                                uint32_t* packed, uint16_t* scales, uint16_t* biases, cudaStream_t s,
                                const QdaRowMap* map, bool pdl) {
  static const QdaRowMap kIdentity = {};
  const QdaRowMap& m = map ? *map : kIdentity;
  const bool f16 = in_dtype == QDA_FP16;
  if (bits == 4) {
    return f16 ? qda::launch_quant<4, true>(x, rows, D, GS, packed, scales, biases, s, m, pdl)
               : qda::launch_quant<4, false>(x, rows, D, GS, packed, scales, biases, s, m, pdl);
  }
  return f16 ? qda::launch_quant<8, true>(x, rows, D, GS, packed, scales, biases, s, m, pdl)
             : qda::launch_quant<8, false>(x, rows, D, GS, packed, scales, biases, s, m, pdl);
}

cudaError_t qda_launch_append_copy(const uint32_t* kp, const uint16_t* ks, const uint16_t* kb, const uint32_t* vp,
                                   const uint16_t* vs, const uint16_t* vb, uint32_t* kpo, uint16_t* kso,
                                   uint16_t* kbo, uint32_t* vpo, uint16_t* vso, uint16_t* vbo, long long rows_old,
                                   int W, int NG, const QdaRowMap& map, cudaStream_t s, bool pdl) {
  if (rows_old <= 0) return cudaSuccess;
  int max_n = 0;
  for (int b = 0; b < map.B; ++b) max_n = std::max(max_n, map.n_old[b]);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((max_n + qda::kAppendRows - 1) / qda::kAppendRows),
                     (unsigned)std::min(map.B * map.Hkv, 65535));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, qda::qda_append_copy_kernel, kp, ks, kb, vp, vs, vb, kpo, kso, kbo, vpo, vso, vbo, W,
                            NG, map);
}
