// Affine-quantized weight GEMV, streamed form (sm_103a): the same product as qda_gemv.cu,
//     y[t, n] = sum_k x[t, k] * (scale[n, k / GS] * code[n, k] + bias[n, k / GS]),   t < T <= 4
// (maya-mac mlx_kernels.py, _linear_kernel), for three or four input rows (four of 4-bit codes) and K <= 4096.
//
// The exact code conversion and the packed FMAs cost about two instructions per code and input row, so with three
// or four input rows the instruction issue, not the stream, sets the time of this product on GB300. This form keeps
// each lane's x values in registers for the whole kernel (the direct-load kernel re-reads its x slice every step)
// and streams each CTA's contiguous block of rows (codes, scales and biases: three 1-D bulk copies per chunk of
// rows) through a shared-memory ring several chunks deep, filled by one producer warp, so the consumer warps issue
// only the arithmetic. For one or two input rows (three of 4-bit codes) the direct-load kernel, with three times
// the warps per SM, was measured faster and is used instead.
//
// Eight consumer warps split a chunk two ways: KW K-slices times RW = 8 / KW row groups, KW the fewest whose x
// values fit a lane. A K-slice is a fixed set of 512-element steps of K (step s belongs to slice s % KW), and each
// lane owns 16 elements of each of its steps, so a lane's x values never change: they are loaded once, as floats,
// into registers (16 * T per step, at most 64). Per row a lane takes its 16 codes per step (one 16-byte or 8-byte
// shared load), turns them into exact floats (byte permute to 2^23 + code, minus 2^23), forms the factored dot
// s * sum(x * code) + b * sum(x) with packed f32x2 FMAs, and the warp adds its lanes by shuffles. The KW slice sums
// of a row meet in shared memory and are added in slice order, so every output is the same from run to run.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qda_split.cuh"

namespace qda {

constexpr int kRingConsumers = 8;                         // consumer warps
constexpr int kRingThreads = (kRingConsumers + 1) * 32;   // + the producer warp
constexpr int kRingRowAlign = 8;                          // chunks start on multiples of 8 rows
constexpr int kRingMaxStages = 8;
constexpr size_t kRingSmemBudget = 227 * 1024;

struct QgemvRingParams {
  const uint16_t* x;          // [T, K] bf16 / fp16
  const uint32_t* wp;         // [N, K * bits / 32] packed codes
  const uint16_t* ws;         // [N, K / GS] scales
  const uint16_t* wb;         // [N, K / GS] biases
  void* y;                    // [T, N] output dtype
  unsigned int* err;          // device error word
  int N, K, GS, NG, f16, out;
  int steps;                  // K / 512
  int kw, rw;                 // K-slices and row groups of the consumer warps (kw * rw = consumer warps)
  int chunk_rows;             // rows per ring slot (a multiple of 8)
  int stages;
  int num_ctas;
  long long blocks;           // ceil(N / 8): CTA c streams blocks [c * blocks / num_ctas, (c + 1) * blocks / num_ctas)
  size_t code_bytes;          // chunk_rows * K * bits / 8
  size_t sc_bytes;            // chunk_rows * NG * 2, rounded up to 16
  size_t slot_bytes;          // code_bytes + 2 * sc_bytes
  size_t ring0;               // offset of slot 0 in shared memory
};

// Bounded wait on a barrier phase taken by lane 0, its result shared with the warp (warp-uniform control flow).
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort, err, 1u);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int OUT>
__device__ __forceinline__ void ring_store(void* y, size_t idx, float v) {
  if constexpr (OUT == QDA_FP32) {
    static_cast<float*>(y)[idx] = v;
  } else if constexpr (OUT == QDA_BF16) {
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(y)[idx] = __float2half_rn(v);
  }
}

// The 16 codes of one lane's piece as 8 exact float pairs (code 2i, code 2i + 1).
template <int BITS>
__device__ __forceinline__ void piece_codes(const unsigned char* src, float2 (&c)[8]) {
  const float2 off = make_float2(-8388608.0f, -8388608.0f);
  if constexpr (BITS == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int j = 0; j < 2; ++j)
        c[2 * k + j] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7650u | (2 * j))),
                                              __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7651u | (2 * j)))),
                                  off);
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t lo = w[k] & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6 of the word in bytes 0..3
      const uint32_t hi = (w[k] >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
#pragma unroll
      for (int j = 0; j < 4; ++j)
        c[4 * k + j] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7650u | j)),
                                              __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7650u | j))),
                                  off);
    }
  }
}

// T input rows, SPW steps per K-slice at most (T * SPW <= 4: 16 * T * SPW x values per lane in registers).
template <int BITS, int T, int SPW, int OUT>
__global__ void __launch_bounds__(kRingThreads, 1) qda_qgemv_ring_kernel(const __grid_constant__ QgemvRingParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);     // [stages] slot landed
  uint64_t* empty = full + kRingMaxStages;                // [stages] slot read by the eight consumer warps
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kRingMaxStages);
  float* part = reinterpret_cast<float*>(smem + 16 * kRingMaxStages + 16);   // [2][chunk_rows][kw][T]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long b0 = (long long)blockIdx.x * p.blocks / p.num_ctas;
  const long long b1 = (long long)(blockIdx.x + 1) * p.blocks / p.num_ctas;
  const int n_beg = (int)(b0 * kRingRowAlign);
  const int n_end = (int)min(b1 * kRingRowAlign, (long long)p.N);
  const int RB = p.K * BITS / 8;   // code bytes per row
  const int CR = p.chunk_rows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRingConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (n_beg >= n_end) return;
  const int chunks = (n_end - n_beg + CR - 1) / CR;

  if (warp == kRingConsumers) {
    // ------------------------------------------------------------------------------------ producer warp
    const uint64_t pol = policy_evict_first();
    int i = 0;
    for (; i < chunks; ++i) {
      const int s = i % p.stages;
      if (i >= p.stages && !ring_wait(&empty[s], ((i / p.stages) - 1) & 1, abort_flag, p.err)) break;
      const int n0 = n_beg + i * CR, rows = min(CR, n_end - n0);
      unsigned char* slot = smem + p.ring0 + (size_t)s * p.slot_bytes;
      const uint32_t cbytes = (uint32_t)rows * RB;
      const uint32_t sbytes = (uint32_t)rows * p.NG * 2, s16 = sbytes & ~15u;
      if (!in_bounds(cbytes <= p.code_bytes && sbytes <= p.sc_bytes && n0 + rows <= p.N, p.err)) {
        if (lane == 0) mbar_arrive_expect_tx(&full[s], 0);
        continue;
      }
      if (lane == 0) {
        if (s16 != sbytes) {   // the matrix's last < 16 bytes of scales and biases: plain loads, published by
                               // the arrive
          const uint16_t* srcs[2] = {p.ws, p.wb};
          for (int a = 0; a < 2; ++a) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(slot + p.code_bytes + a * p.sc_bytes + s16);
            const uint16_t* src = srcs[a] + (size_t)n0 * p.NG + s16 / 2;
            for (uint32_t k = 0; k < (sbytes - s16) / 2; ++k) dst[k] = src[k];
          }
        }
        mbar_arrive_expect_tx(&full[s], cbytes + 2 * s16);
      }
      __syncwarp();
      if (lane == 0) {
        bulk_g2s(slot, reinterpret_cast<const unsigned char*>(p.wp) + (size_t)n0 * RB, cbytes, &full[s], pol);
      } else if (lane < 3 && s16) {
        const uint16_t* src = lane == 1 ? p.ws : p.wb;
        bulk_g2s(slot + p.code_bytes + (lane - 1) * p.sc_bytes, src + (size_t)n0 * p.NG, s16, &full[s], pol);
      }
    }
    if (lane == 0)   // every issued copy lands before the CTA exits
      for (int j = (i > p.stages ? i - p.stages : 0); j < i; ++j)
        mbar_wait_drain(&full[j % p.stages], (j / p.stages) & 1, p.err);
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------------------------------- consumer warps
  const int ks = warp % p.kw, rg = warp / p.kw;   // this warp's K-slice and row group
  // x of this lane's pieces: step ks + kw * j, elements 512 * step + 16 * lane .. + 15, and their sums
  float2 xv[SPW][T][8];
  float xs[SPW][T];
  int g_of[SPW];   // group of each piece
  int nsteps = 0;
#pragma unroll
  for (int j = 0; j < SPW; ++j) {
    const int st = ks + p.kw * j;
    const bool live = st < p.steps;
    nsteps += live ? 1 : 0;
    const int k0 = 512 * st + 16 * lane;
    g_of[j] = live ? k0 / p.GS : 0;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint4 a = make_uint4(0u, 0u, 0u, 0u);
        if (live) a = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.K + k0) + q);
        const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xv[j][t][4 * q + i] = make_float2(half_bits_to_float_rt(u[i] & 0xFFFFu, p.f16 != 0),
                                            half_bits_to_float_rt(u[i] >> 16, p.f16 != 0));
          sum += xv[j][t][4 * q + i].x + xv[j][t][4 * q + i].y;
        }
      }
      xs[j][t] = sum;
    }
  }

  bool ok = true;
  for (int i = 0; i < chunks; ++i) {
    const int s = i % p.stages;
    const int n0 = n_beg + i * CR, rows = min(CR, n_end - n0);
    ok = ok && ring_wait(&full[s], (i / p.stages) & 1, abort_flag, p.err);
    const unsigned char* slot = smem + p.ring0 + (size_t)s * p.slot_bytes;
    const uint16_t* sS = reinterpret_cast<const uint16_t*>(slot + p.code_bytes);
    const uint16_t* sB = reinterpret_cast<const uint16_t*>(slot + p.code_bytes + p.sc_bytes);
    float* pb = part + (size_t)(i & 1) * CR * p.kw * T;
    for (int r = rg; ok && r < rows; r += p.rw) {
      float acc[T];
#pragma unroll
      for (int t = 0; t < T; ++t) acc[t] = 0.f;
#pragma unroll
      for (int j = 0; j < SPW; ++j) {
        if (j < nsteps) {
          const int st = ks + p.kw * j;
          float2 c[8];
          piece_codes<BITS>(slot + (size_t)r * RB + (512 * st + 16 * lane) * BITS / 8, c);
          const float sc = half_bits_to_float_rt(sS[r * p.NG + g_of[j]], p.f16 != 0);
          const float bi = half_bits_to_float_rt(sB[r * p.NG + g_of[j]], p.f16 != 0);
#pragma unroll
          for (int t = 0; t < T; ++t) {
            float2 d = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 8; ++q) d = __ffma2_rn(c[q], xv[j][t][q], d);
            acc[t] = fmaf(sc, d.x + d.y, fmaf(bi, xs[j][t], acc[t]));
          }
        }
      }
#pragma unroll
      for (int t = 0; t < T; ++t) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
      }
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < T; ++t) pb[((size_t)r * p.kw + ks) * T + t] = acc[t];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    // every slice sum of this chunk is written: the rows' outputs, slices added in order
    named_barrier_sync(1, kRingConsumers * 32);
    // output idx goes to warp idx % 8, lane idx / 8 (no warp takes them all)
    for (int idx = lane * kRingConsumers + warp; idx < rows * T; idx += kRingConsumers * 32) {
      const int r = idx / T, t = idx - r * T;
      float v = 0.f;
      for (int k = 0; k < p.kw; ++k) v += pb[((size_t)r * p.kw + k) * T + t];
      if (ok) ring_store<OUT>(p.y, (size_t)t * p.N + n0 + r, v);
    }
  }
}

// The instances built: three or four input rows, one step per K-slice (the shapes where the streamed form was
// measured faster than the direct-load kernel).
template <int BITS, int OUT, typename Fn>
cudaError_t with_ring_kernel(int T, int spw, Fn&& f) {
  if (spw == 1 && T == 3) return f(qda_qgemv_ring_kernel<BITS, 3, 1, OUT>);
  if (spw == 1 && T == 4) return f(qda_qgemv_ring_kernel<BITS, 4, 1, OUT>);
  return cudaErrorNotSupported;
}

}  // namespace qda

cudaError_t qda_launch_qgemv_ring(const uint16_t* x, const uint32_t* wp, const uint16_t* ws, const uint16_t* wb,
                                  void* y, int T, int N, int K, int GS, int bits, int f16, int out, int sms,
                                  unsigned int* err, cudaStream_t s, bool* launched) {
  using namespace qda;
  *launched = false;
  const long long RB = (long long)K * bits / 8;
  // one or two input rows (three of 4-bit codes): the direct-load kernel was measured faster (both forms issue about
  // the same instructions per code, and it has three times the warps per SM to issue them)
  if (K % 512 != 0 || RB * kRingRowAlign > 64 * 1024 || T < (bits == 8 ? 3 : 4) || T > 4) return cudaSuccess;
  QgemvRingParams p = {};
  p.x = x; p.wp = wp; p.ws = ws; p.wb = wb; p.y = y; p.err = err;
  p.N = N; p.K = K; p.GS = GS; p.NG = K / GS; p.f16 = f16; p.out = out;
  p.steps = K / 512;
  // the fewest K-slices whose x values fit a lane (16 * T per step, 64 at most): each slice sum is one cross-lane
  // reduction and one shared-memory partial per row, so longer slices spread that cost over more codes
  p.kw = 1;
  while (p.kw < kRingConsumers && T * ((p.steps + p.kw - 1) / p.kw) > 4) p.kw *= 2;
  p.rw = kRingConsumers / p.kw;
  const int spw = (p.steps + p.kw - 1) / p.kw;
  if (spw != 1) return cudaSuccess;
  // about 32 KB of codes per slot, whole 8-row blocks
  long long cr = std::max<long long>(1, 32768 / (RB * kRingRowAlign)) * kRingRowAlign;
  cr = std::min<long long>(cr, 64);
  p.chunk_rows = (int)cr;
  p.code_bytes = (size_t)(cr * RB);
  p.sc_bytes = ((size_t)cr * p.NG * 2 + 15) & ~(size_t)15;
  p.slot_bytes = p.code_bytes + 2 * p.sc_bytes;
  const size_t part_bytes = 2 * (size_t)cr * p.kw * T * sizeof(float);
  p.ring0 = (16 * kRingMaxStages + 16 + part_bytes + 127) & ~(size_t)127;
  const long long st = (long long)(kRingSmemBudget - p.ring0) / (long long)p.slot_bytes;
  if (st < 2) return cudaSuccess;
  p.stages = (int)std::min<long long>(kRingMaxStages, st);
  const size_t smem = p.ring0 + (size_t)p.stages * p.slot_bytes;
  p.blocks = (N + kRingRowAlign - 1) / kRingRowAlign;
  p.num_ctas = (int)std::min<long long>(p.blocks, sms);
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_limit(kern, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.num_ctas), kRingThreads, smem, s, p);
  };
  auto dispatch = [&](auto bits_tag) -> cudaError_t {
    constexpr int B = decltype(bits_tag)::value;
    if (out == QDA_BF16) return with_ring_kernel<B, QDA_BF16>(T, spw, launch);
    if (out == QDA_FP16) return with_ring_kernel<B, QDA_FP16>(T, spw, launch);
    return with_ring_kernel<B, QDA_FP32>(T, spw, launch);
  };
  *launched = true;
  return bits == 8 ? dispatch(std::integral_constant<int, 8>()) : dispatch(std::integral_constant<int, 4>());
}
