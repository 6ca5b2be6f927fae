// Host side of libqdecode_attn: argument checks, the launch plan, workspace handling and the C entry points.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include <cuda.h>

#include "qda_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kMinRowsPerCta = 128;
constexpr long long kMaxCtas = 4096;   // plan cap: CTA row ranges use a 64-bit magic division exact up to here

thread_local int t_last_cuda_error = 0;
thread_local void* t_split_event = nullptr;
std::atomic<int> g_force_splits{0};
std::atomic<int> g_stall_chunk{-1};
std::atomic<long long> g_calls{0};

__device__ unsigned int g_device_err;

struct DeviceState {
  std::mutex mu;
  bool init = false;
  int num_sms = 0;
  unsigned int* err = nullptr;      // address of g_device_err on this device
  void* ws = nullptr;               // library-owned workspace
  size_t ws_bytes = 0;
  std::vector<void*> retired;       // outgrown workspaces, kept allocated until the process ends
  void* user_ws = nullptr;          // caller-installed workspace
  size_t user_ws_bytes = 0;
  std::map<std::tuple<int, int, int, int, int, size_t>, int> occupancy;
};
DeviceState g_dev[kMaxDevices];

// Staging of the host-buffer entry point on one device: two sets of device buffers used in turn, so that one call's
// host->device copies (on the library's copy stream) overlap the previous call's kernels (on the caller's stream).
struct HostStage {
  std::mutex mu;
  cudaStream_t copy = nullptr;
  cudaEvent_t copied[2] = {nullptr, nullptr};    // set i holds this call's inputs
  cudaEvent_t released[2] = {nullptr, nullptr};  // the last work that read set i (kernels, output copy) is done
  void* buf[2] = {nullptr, nullptr};
  size_t bytes[2] = {0, 0};
  int turn = 0;
};
HostStage g_stage[kMaxDevices];

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return QDA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pure host checks of the shape (no pointers): the support predicate of mlx-bun fused-decode-kernel.ts
// (fusedDecodeKernelSupported), widened to B >= 1 sequences, any H % Hkv == 0, fp16 or bf16 input and L query
// positions per sequence.
int check_shape(int B, int L, int H, int Hkv, const int32_t* N, int D, int GS, int bits) {
  if (N == nullptr) return QDA_ERR_INVALID;
  if (B < 1 || L < 1 || H < 1 || Hkv < 1 || D < 1 || GS < 1) return QDA_ERR_INVALID;
  if (H % Hkv != 0) return QDA_ERR_INVALID;
  for (int b = 0; b < B && b <= QDA_MAX_B; ++b)
    if (N[b] < L) return QDA_ERR_INVALID;
  if (bits != 4 && bits != 8) return QDA_ERR_UNSUPPORTED;
  if (GS != 32 && GS != 64 && GS != 128) return QDA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256 && D != 512) return QDA_ERR_UNSUPPORTED;
  if (D % GS != 0) return QDA_ERR_UNSUPPORTED;
  if (B > QDA_MAX_B) return QDA_ERR_UNSUPPORTED;
  if (L > QDA_MAX_L || (H / Hkv) * L > QDA_MAX_NREP) return QDA_ERR_UNSUPPORTED;
  long long total = 0;
  for (int b = 0; b < B; ++b) total += N[b];
  if (total > (1LL << 31) - 1) return QDA_ERR_UNSUPPORTED;   // sequence offsets are int32
  return QDA_OK;
}

int check_dtype(int dtype, int* in, int* out) {
  const int i = dtype & 0xff, o = (dtype >> 8) & 0xff;
  if ((dtype >> 16) != 0) return QDA_ERR_INVALID;
  if (i != QDA_BF16 && i != QDA_FP16) return QDA_ERR_INVALID;
  if (o != 0 && o != QDA_BF16 && o != QDA_FP16 && o != QDA_FP32) return QDA_ERR_INVALID;
  *in = i;
  *out = o == 0 ? i : o;
  return QDA_OK;
}

// The split kernel's configuration for one shape.
struct Variant {
  int W, nh, hc, heads_pad, NG, tile, stages;   // words per row, heads per CTA, head chunks, ..., ring stages
  size_t smem;
  bool tc = false;                              // the tensor-core split kernel (qda_tc.cuh)
  int threads = QDA_THREADS;
  int kstages = 0;                              // tensor-core kernel: K-ring depth (stages: V-ring depth)
};

constexpr size_t kSmemBudget = 112 * 1024;   // two CTAs per SM

// Rows per warp block of the lean kernel (its Split2Geom<...>::R).
int split2_rows(int D, int nh) { return nh == 4 ? 8 : 16; }

// nrep: query heads served per KV head (H / Hkv, times L for multi-query decode). D is one of 64, 128, 256, 512.
Variant pick_variant(int nrep, int D, int GS, int bits) {
  Variant v;
  v.W = D * bits / 32;
  v.NG = D / GS;
  v.nh = (nrep <= 2 || D == 512) ? 2 : 4;   // D = 512 takes heads two at a time (register budget)
  v.hc = (nrep + v.nh - 1) / v.nh;
  v.heads_pad = v.hc * v.nh;
  const int R = split2_rows(D, v.nh);
  v.tile = QDA_SPLIT2_TILE;   // warps take TILE / R blocks of a chunk in turn (the kernel's constant tile)
  const QdaSmemLayout L = qda_smem_layout(v.tile, 1, v.W, v.NG, v.nh, D);
  const size_t scratch = (size_t)QDA_NW * split2_scratch_floats(R, v.NG, v.nh) * 4;
  const size_t comb = (size_t)QDA_NW * v.nh * D * 4 + (size_t)QDA_NW * v.nh * 2 * 4;
  const size_t tail = std::max(scratch, comb);
  long long st = ((long long)kSmemBudget - (long long)L.stage0 - (long long)tail) / (long long)L.stage_bytes;
  v.stages = (int)std::max(2LL, std::min(8LL, st));
  v.smem = L.stage0 + (size_t)v.stages * L.stage_bytes + tail;
  return v;
}

constexpr size_t kTcSmemBudget = 227 * 1024;   // one CTA per SM
constexpr long long kTcMaxRows = (1LL << 31) - 2 * QDA_TC_TILE;   // tensor-copy row coordinates are int32

// The tensor-core kernel serves single-query decode of 4-bit caches at D = 128 and 256 with at least two groups
// per row and three or more query heads per KV head (four per CTA); T is the cache's total row count.
bool tc_eligible(int nrep, int D, int GS, int bits, long long T) {
  return bits == 4 && (D == 128 || D == 256) && D / GS >= 2 && nrep >= 3 && T <= kTcMaxRows;
}

Variant pick_tc_variant(int nrep, int D, int GS) {
  Variant v;
  v.tc = true;
  v.threads = QDA_TC_THREADS;
  v.W = D / 8;
  v.NG = D / GS;
  v.nh = 4;
  v.hc = (nrep + 3) / 4;
  v.heads_pad = v.hc * 4;
  v.tile = qda_tc_slot_rows(D);   // the chunk walker's tile: one ring slot (several 128-row MMA tiles)
  // K ring: two slots (one being converted, one in flight); V ring: what shared memory leaves, 2 to 8 slots
  v.kstages = 2;
  const QdaTcLayout L0 = qda_tc_layout(D, 4, v.NG, v.kstages, 0);
  const long long st = ((long long)kTcSmemBudget - (long long)L0.total) / (long long)L0.vstage_bytes;
  v.stages = (int)std::max(2LL, std::min(8LL, st));
  v.smem = qda_tc_layout(D, 4, v.NG, v.kstages, v.stages).total;
  return v;
}

cudaError_t split_occupancy(int bits, int D, bool exact, const Variant& v, int* n) {
  if (v.tc) {
    return exact ? qda_occupancy_tc_x1(D, v.nh, v.NG, v.smem, n) : qda_occupancy_tc_x0(D, v.nh, v.NG, v.smem, n);
  }
  if (bits == 4) {
    return exact ? qda_occupancy_split2_b4_x1(D, v.nh, v.NG, v.smem, n)
                 : qda_occupancy_split2_b4_x0(D, v.nh, v.NG, v.smem, n);
  }
  return exact ? qda_occupancy_split2_b8_x1(D, v.nh, v.NG, v.smem, n)
               : qda_occupancy_split2_b8_x0(D, v.nh, v.NG, v.smem, n);
}

cudaError_t split_launch(int bits, bool exact, const QdaParams& p, const Variant& v, dim3 grid, cudaStream_t s) {
  if (bits == 4) {
    return exact ? qda_launch_split2_b4_x1(p, p.D, v.nh, v.NG, grid, v.smem, s)
                 : qda_launch_split2_b4_x0(p, p.D, v.nh, v.NG, grid, v.smem, s);
  }
  return exact ? qda_launch_split2_b8_x1(p, p.D, v.nh, v.NG, grid, v.smem, s)
               : qda_launch_split2_b8_x0(p, p.D, v.nh, v.NG, grid, v.smem, s);
}

// The plan: one contiguous, equal share of the flattened rows per CTA, as many CTAs as fit on the GPU at once
// (one wave), but no fewer than kMinRowsPerCta rows each. Deterministic in (shape, SM count, occupancy).
void make_plan(int B, int Hkv, const int32_t* N, int D, int num_sms, int ctas_per_sm, const Variant& v,
               qda_plan* plan) {
  long long sumN = 0;
  for (int b = 0; b < B; ++b) sumN += N[b];
  const long long T = (long long)Hkv * sumN;
  const int units = B * Hkv;
  long long target = std::max(1LL, (long long)num_sms * std::max(1, ctas_per_sm) / v.hc);
  long long by_rows = std::max(1LL, (T + kMinRowsPerCta - 1) / kMinRowsPerCta);
  long long C = std::min(target, by_rows);
  const int forced = g_force_splits.load();
  if (forced > 0) C = forced;
  C = std::min<long long>(C, kMaxCtas);
  plan->num_ctas = (int)C;
  plan->head_chunks = v.hc;
  plan->heads_per_cta = v.nh;
  plan->tile_rows = v.tile;
  plan->stages = v.stages;
  plan->threads = v.threads;
  plan->units = units;
  plan->smem_bytes = (int)v.smem;
  plan->total_rows = T;
  plan->slots = C + units;
  const size_t o_bytes = (size_t)plan->slots * v.heads_pad * D * sizeof(float);
  const size_t ml_bytes = (size_t)plan->slots * v.heads_pad * 2 * sizeof(float);
  plan->workspace_bytes = ((o_bytes + 255) & ~(size_t)255) + ml_bytes;
}

DeviceState* device_state(int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    t_last_cuda_error = (int)e;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceState& d = g_dev[dev];
  std::lock_guard<std::mutex> lock(d.mu);
  if (!d.init) {
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_device_err)) != cudaSuccess) {
      t_last_cuda_error = (int)e;
      return nullptr;
    }
    d.init = true;
  }
  *dev_out = dev;
  return &d;
}

int occupancy_for(DeviceState& d, int bits, int D, bool exact, const Variant& v, int* n) {
  std::lock_guard<std::mutex> lock(d.mu);
  auto key = std::make_tuple(bits + 16 * (int)exact, D, (int)v.tc, v.nh, v.NG, v.smem);
  auto it = d.occupancy.find(key);
  if (it != d.occupancy.end()) {
    *n = it->second;
    return QDA_OK;
  }
  cudaError_t e = split_occupancy(bits, D, exact, v, n);
  if (e != cudaSuccess) return cuda_fail(e);
  if (*n < 1) *n = 1;
  d.occupancy[key] = *n;
  return QDA_OK;
}

// ------------------------------------------------------------------------------------------------------------
// Scratch of the allocation-free entry point: its partial results live in this fixed device array instead of a
// cudaMalloc'ed workspace. Host code must not pass the array's name to a kernel (on the host it names a stand-in, not device
// memory): the device address is looked up once per device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) unsigned char g_qda_static_scratch[QDA_STATIC_SCRATCH_BYTES];
std::mutex g_static_mu;
void* g_static_scratch_addr[kMaxDevices] = {};

// The 2-D tensor map of a cache's K codes for the tensor-core kernel: rows of D / 2 bytes, boxes of 256 rows by
// min(D / 2, 128) bytes, 16-byte chunks swizzled within 128-byte (64-byte at D = 128) rows so that one thread per
// row reads shared memory without bank conflicts. cuTensorMapEncodeTiled comes from the driver through the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encode_k_map(const uint32_t* k_packed, int D, long long rows, CUtensorMap* map) {
  static EncodeTiledFn fn = nullptr;
  static cudaError_t fn_status = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    fn_status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (fn_status == cudaSuccess && (q != cudaDriverEntryPointSuccess || f == nullptr))
      fn_status = cudaErrorSymbolNotFound;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  if (fn_status != cudaSuccess) return fn_status;
  const cuuint64_t rb = (cuuint64_t)D / 2;
  const cuuint64_t dims[2] = {rb, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {rb};
  const cuuint32_t box[2] = {(cuuint32_t)std::min<cuuint64_t>(rb, 128), 256};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(k_packed), dims, strides, box,
                        elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        rb >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The split kernel a call takes: the tensor-core kernel for single-query decode where it applies, else the lean
// CUDA-core kernel (every shape, multi-query decode and the compat form).
Variant choose_variant(int B, int L, int nrep, int Hkv, const int32_t* N, int D, int GS, int bits, bool compat) {
  long long T = 0;
  for (int b = 0; b < B; ++b) T += (long long)N[b] * Hkv;
  if (L == 1 && !compat && tc_eligible(nrep, D, GS, bits, T)) return pick_tc_variant(nrep, D, GS);
  return pick_variant(nrep * L, D, GS, bits);
}

int plan_impl(int B, int L, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int num_sms, int ctas_per_sm,
              qda_plan* plan) {
  if (plan == nullptr) return QDA_ERR_INVALID;
  int st = check_shape(B, L, H, Hkv, N, D, GS, bits);
  if (st != QDA_OK) return st;
  const Variant v = choose_variant(B, L, H / Hkv, Hkv, N, D, GS, bits, false);
  if (num_sms <= 0 || ctas_per_sm <= 0) {
    int dev;
    DeviceState* d = device_state(&dev);
    if (d == nullptr) return QDA_ERR_CUDA;
    if (num_sms <= 0) num_sms = d->num_sms;
    if (ctas_per_sm <= 0) {
      // the input dtype does not change the kernel's resources; bf16 stands for both
      st = occupancy_for(*d, bits, D, false, v, &ctas_per_sm);
      if (st != QDA_OK) return st;
    }
  }
  make_plan(B, Hkv, N, D, num_sms, ctas_per_sm, v, plan);
  return QDA_OK;
}

// Where a call's partial results live.
enum class Scratch { kWorkspace, kStatic };

// Every decode entry point: checks, plan, scratch, parameters, the split and merge launches.
// compat: the two-pass form with the pages' rounding points (one query position).
int run_call(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
             const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out, int B, int L, int H,
             int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream, Scratch where,
             bool compat = false) {
  if (!q || !k_packed || !k_scales || !k_biases || !v_packed || !v_scales || !v_biases || !out)
    return QDA_ERR_INVALID;
  int in_dt, out_dt;
  int st = check_dtype(dtype, &in_dt, &out_dt);
  if (st != QDA_OK) return st;
  st = check_shape(B, L, H, Hkv, N, D, GS, bits);
  if (st != QDA_OK) return st;
  const void* ptrs[8] = {q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, out};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return QDA_ERR_ALIGN;

  const int nrep = H / Hkv;
  if (compat && L != 1) return QDA_ERR_UNSUPPORTED;
  const Variant v = choose_variant(B, L, nrep, Hkv, N, D, GS, bits, compat);
  int dev;
  DeviceState* d = device_state(&dev);
  if (d == nullptr) return QDA_ERR_CUDA;
  const bool exact = out_dt == QDA_FP32;
  int occ = 1;
  st = occupancy_for(*d, bits, D, exact, v, &occ);
  if (st != QDA_OK) return st;
  qda_plan plan;
  make_plan(B, Hkv, N, D, d->num_sms, occ, v, &plan);

  void* ws = nullptr;
  if (where == Scratch::kStatic) {
    if (plan.workspace_bytes > (size_t)QDA_STATIC_SCRATCH_BYTES) return QDA_ERR_SCRATCH;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_scratch_addr[dev] == nullptr) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_qda_static_scratch);
      if (e != cudaSuccess) return cuda_fail(e);
      g_static_scratch_addr[dev] = ptr;
    }
    ws = g_static_scratch_addr[dev];
  } else {
    std::lock_guard<std::mutex> lock(d->mu);
    if (d->user_ws != nullptr) {
      if (d->user_ws_bytes < plan.workspace_bytes) return QDA_ERR_WORKSPACE;
      ws = d->user_ws;
    } else {
      if (d->ws_bytes < plan.workspace_bytes) {
        // grow (at least doubling); the smaller buffer is retired, not freed: a CUDA graph captured earlier or a
        // launch another thread is about to make may still write to it
        const size_t want = std::max({plan.workspace_bytes, 2 * d->ws_bytes, (size_t)1 << 20});
        void* grown = nullptr;
        cudaError_t e = cudaMalloc(&grown, want);
        if (e != cudaSuccess) return cuda_fail(e);
        if (d->ws != nullptr) d->retired.push_back(d->ws);
        d->ws = grown;
        d->ws_bytes = want;
      }
      ws = d->ws;
    }
  }

  QdaParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.kp = k_packed;
  p.ks = static_cast<const uint16_t*>(k_scales);
  p.kb = static_cast<const uint16_t*>(k_biases);
  p.vp = v_packed;
  p.vs = static_cast<const uint16_t*>(v_scales);
  p.vb = static_cast<const uint16_t*>(v_biases);
  const size_t o_bytes = (size_t)plan.slots * v.heads_pad * D * sizeof(float);
  p.part_o = static_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + ((o_bytes + 255) & ~(size_t)255));
  p.err = d->err;
  p.total_rows = plan.total_rows;
  p.cta_magic = ~0ULL / (unsigned long long)plan.num_ctas + 1ULL;
  p.B = B;
  p.L = L;
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.GS = GS;
  p.NG = v.NG;
  p.W = v.W;
  p.nrep = nrep;
  p.heads_pad = v.heads_pad;
  p.head_chunks = v.hc;
  p.num_ctas = plan.num_ctas;
  p.tile_rows = v.tile;
  p.stages = v.stages;
  p.kstages = v.kstages;
  p.tile_shift = 0;
  while ((1 << p.tile_shift) < v.tile) ++p.tile_shift;
  p.f16 = in_dt == QDA_FP16 ? 1 : 0;
  p.stall_chunk = g_stall_chunk.load();
  // scores in log2 units, except in the compat form, which rounds them in natural units first
  p.qscale = (compat ? 1.0f : 1.4426950408889634f) / sqrtf((float)D);
  p.seq_off[0] = 0;
  for (int b = 0; b < B; ++b) p.seq_off[b + 1] = p.seq_off[b] + N[b];

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid((unsigned)plan.num_ctas * (unsigned)v.hc);
  cudaError_t e;
  // the lean split kernel launches behind the previous kernel with programmatic dependent launch only in the compat
  // form's second pass (behind its first): as a call's first launch the attribute measured 0.2 us slower at 8k
  p.launch_pdl = 0;
  if (compat) {
    p.mode = 2;   // pass A: K only, per-range statistics of the rounded scores
    p.k_only = 1;
    e = split_launch(bits, exact, p, v, grid, s);
    if (e != cudaSuccess) return cuda_fail(e);
    p.mode = 3;   // pass B: normalised, rounded probabilities times V
    p.k_only = 0;
    p.compat = 1;
    p.launch_pdl = 1;
  } else {
    p.mode = L > 1 ? 1 : 0;
  }
  if (v.tc) {
    CUtensorMap tmk;
    e = encode_k_map(k_packed, D, plan.total_rows, &tmk);
    if (e != cudaSuccess) return cuda_fail(e);
    e = exact ? qda_launch_tc_x1(p, &tmk, D, v.nh, v.NG, grid, v.smem, s)
              : qda_launch_tc_x0(p, &tmk, D, v.nh, v.NG, grid, v.smem, s);
  } else {
    e = split_launch(bits, exact, p, v, grid, s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  const bool use_event = t_split_event != nullptr && where == Scratch::kWorkspace;
  if (use_event) {
    e = cudaEventRecord(static_cast<cudaEvent_t>(t_split_event), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  // a head whose partials span many slots is merged by D / 64 CTAs (one per 64 values) instead of one: about
  // slots * D / 2048 dependent slot loads per thread group of one CTA, more than 6 leave the merge latency-bound
  int max_n = 0;
  for (int b = 0; b < B; ++b) max_n = std::max(max_n, (int)N[b]);
  const long long slots = (long long)max_n * plan.num_ctas / std::max(1LL, plan.total_rows) + 2;
  const int slices = (D >= 128 && slots * D > 6LL * 2048) ? D / 64 : 1;
  e = qda_launch_merge(p, out, out_dt, !use_event, slices, d->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e);
  g_calls.fetch_add(1);
  return QDA_OK;
}

}  // namespace

int qda_cuda_fail(cudaError_t e) { return cuda_fail(e); }

extern "C" {

int qdecode_attn_plan(int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int num_sms,
                      int ctas_per_sm, qda_plan* plan) {
  return plan_impl(B, 1, H, Hkv, N, D, GS, bits, num_sms, ctas_per_sm, plan);
}

int qdecode_attn_multi_plan(int B, int L, int H, int Hkv, const int32_t* N, int D, int GS, int bits, int num_sms,
                            int ctas_per_sm, qda_plan* plan) {
  return plan_impl(B, L, H, Hkv, N, D, GS, bits, num_sms, ctas_per_sm, plan);
}

int qdecode_attn_workspace_bytes(int B, int H, int Hkv, const int32_t* N, int D, int GS, int bits, size_t* bytes) {
  if (bytes == nullptr) return QDA_ERR_INVALID;
  int st = check_shape(B, 1, H, Hkv, N, D, GS, bits);
  if (st != QDA_OK) return st;
  int dev;
  DeviceState* d = device_state(&dev);
  if (d == nullptr) return QDA_ERR_CUDA;
  // the largest need of every call of this shape: qdecode_attn (tensor-core or lean kernel) and qdecode_attn_compat,
  // each with 16-bit or fp32 output (the output form selects a kernel instance whose occupancy can differ)
  const int nrep = H / Hkv;
  const Variant vs[2] = {choose_variant(B, 1, nrep, Hkv, N, D, GS, bits, false), pick_variant(nrep, D, GS, bits)};
  size_t most = 0;
  for (const Variant& v : vs) {
    for (int exact = 0; exact < 2; ++exact) {
      int occ = 1;
      st = occupancy_for(*d, bits, D, exact != 0, v, &occ);
      if (st != QDA_OK) return st;
      qda_plan plan;
      make_plan(B, Hkv, N, D, d->num_sms, occ, v, &plan);
      most = std::max(most, plan.workspace_bytes);
    }
  }
  *bytes = most;
  return QDA_OK;
}

int qdecode_attn_set_workspace(void* ptr, size_t bytes) {
  if (ptr != nullptr && !aligned16(ptr)) return QDA_ERR_ALIGN;
  int dev;
  DeviceState* d = device_state(&dev);
  if (d == nullptr) return QDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(d->mu);
  d->user_ws = ptr;
  d->user_ws_bytes = ptr ? bytes : 0;
  return QDA_OK;
}

int qdecode_attn_debug_force_splits(int num_ctas) {
  if (num_ctas < 0) return QDA_ERR_INVALID;
  g_force_splits.store(num_ctas);
  return QDA_OK;
}

int qdecode_attn_debug_stall_chunk(int chunk) {
  g_stall_chunk.store(chunk < 0 ? -1 : chunk);
  return QDA_OK;
}

int qdecode_attn_set_split_event(void* event) {
  t_split_event = event;
  return QDA_OK;
}

int qdecode_attn(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                 const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out, int B, int H,
                 int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream) {
  return run_call(q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, out, B, 1, H, Hkv, N, D, GS, bits,
                  dtype, stream, Scratch::kWorkspace);
}

int qdecode_attn_multi(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                       const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out, int B, int L,
                       int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream) {
  return run_call(q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, out, B, L, H, Hkv, N, D, GS, bits,
                  dtype, stream, Scratch::kWorkspace);
}

int qdecode_attn_compat(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                        const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out, int B,
                        int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream) {
  return run_call(q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, out, B, 1, H, Hkv, N, D, GS, bits,
                  dtype, stream, Scratch::kWorkspace, true);
}

// The allocation-free entry point: partial results in the fixed device array above, never in an allocation.
int qdecode_attn_noalloc(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                         const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out, int B,
                         int H, int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream) {
  return run_call(q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, out, B, 1, H, Hkv, N, D, GS, bits,
                  dtype, stream, Scratch::kStatic);
}

// Host buffers in and out: stage the inputs on the device, decode, copy the output back (all asynchronous).
int qdecode_attn_host(const void* q, const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                      const uint32_t* v_packed, const void* v_scales, const void* v_biases, void* out, int B, int H,
                      int Hkv, const int32_t* N, int D, int GS, int bits, int dtype, void* stream) {
  if (!q || !k_packed || !k_scales || !k_biases || !v_packed || !v_scales || !v_biases || !out)
    return QDA_ERR_INVALID;
  int in_dt, out_dt;
  int st = check_dtype(dtype, &in_dt, &out_dt);
  if (st != QDA_OK) return st;
  st = check_shape(B, 1, H, Hkv, N, D, GS, bits);
  if (st != QDA_OK) return st;
  int dev;
  DeviceState* d = device_state(&dev);
  if (d == nullptr) return QDA_ERR_CUDA;
  long long T = 0;
  for (int b = 0; b < B; ++b) T += (long long)N[b] * Hkv;
  const size_t in_size = 2, out_size = out_dt == QDA_FP32 ? 4 : 2;
  // q, K codes, K scales, K biases, V codes, V scales, V biases, out; each piece 256-byte aligned in the set
  const size_t sizes[8] = {(size_t)B * H * D * in_size, (size_t)T * (D * bits / 32) * 4, (size_t)T * (D / GS) * 2,
                           (size_t)T * (D / GS) * 2,    (size_t)T * (D * bits / 32) * 4, (size_t)T * (D / GS) * 2,
                           (size_t)T * (D / GS) * 2,    (size_t)B * H * D * out_size};
  size_t offs[9];
  offs[0] = 0;
  for (int i = 0; i < 8; ++i) offs[i + 1] = offs[i] + ((sizes[i] + 255) & ~(size_t)255);
  const void* src[7] = {q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases};
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  HostStage& g = g_stage[dev];
  std::lock_guard<std::mutex> lock(g.mu);
  cudaError_t e;
  if (g.copy == nullptr) {
    if ((e = cudaStreamCreateWithFlags(&g.copy, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
    for (int i = 0; i < 2; ++i) {
      if ((e = cudaEventCreateWithFlags(&g.copied[i], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&g.released[i], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e);
    }
  }
  const int k = g.turn;
  if (g.bytes[k] < offs[8]) {
    // the set may still be read by an earlier call's work: wait for it before freeing
    if ((e = cudaEventSynchronize(g.released[k])) != cudaSuccess) return cuda_fail(e);
    if (g.buf[k] != nullptr) cudaFree(g.buf[k]);
    g.buf[k] = nullptr;
    g.bytes[k] = 0;
    if ((e = cudaMalloc(&g.buf[k], offs[8])) != cudaSuccess) return cuda_fail(e);
    g.bytes[k] = offs[8];
  }
  char* base = static_cast<char*>(g.buf[k]);
  // this set's previous readers are done before its copies overwrite it; then the inputs, then the caller's stream
  // waits for them
  if ((e = cudaStreamWaitEvent(g.copy, g.released[k], 0)) != cudaSuccess) return cuda_fail(e);
  for (int i = 0; i < 7; ++i)
    if ((e = cudaMemcpyAsync(base + offs[i], src[i], sizes[i], cudaMemcpyHostToDevice, g.copy)) != cudaSuccess)
      return cuda_fail(e);
  if ((e = cudaEventRecord(g.copied[k], g.copy)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaStreamWaitEvent(s, g.copied[k], 0)) != cudaSuccess) return cuda_fail(e);
  st = run_call(base + offs[0], reinterpret_cast<const uint32_t*>(base + offs[1]), base + offs[2], base + offs[3],
                reinterpret_cast<const uint32_t*>(base + offs[4]), base + offs[5], base + offs[6], base + offs[7], B,
                1, H, Hkv, N, D, GS, bits, dtype, stream, Scratch::kWorkspace);
  if (st != QDA_OK) return st;
  if ((e = cudaMemcpyAsync(out, base + offs[7], sizes[7], cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaEventRecord(g.released[k], s)) != cudaSuccess) return cuda_fail(e);
  g.turn = k ^ 1;
  return QDA_OK;
}

int qdecode_quantize(const float* x, long long rows, int D, int GS, int bits, int dtype, uint32_t* packed,
                     void* scales, void* biases, void* stream) {
  if (!x || !packed || !scales || !biases) return QDA_ERR_INVALID;
  if (rows < 1 || D < 1 || GS < 1) return QDA_ERR_INVALID;
  int in_dt, out_dt;
  int st = check_dtype(dtype, &in_dt, &out_dt);
  if (st != QDA_OK) return st;
  if (bits != 4 && bits != 8) return QDA_ERR_UNSUPPORTED;
  if (GS != 32 && GS != 64 && GS != 128) return QDA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256 && D != 512) return QDA_ERR_UNSUPPORTED;
  if (D % GS != 0) return QDA_ERR_UNSUPPORTED;
  if (rows > (1LL << 31) * 8 - 8) return QDA_ERR_UNSUPPORTED;
  if (((uintptr_t)x & 15u) || ((uintptr_t)packed & 3u) || ((uintptr_t)scales & 1u) || ((uintptr_t)biases & 1u))
    return QDA_ERR_ALIGN;
  cudaError_t e = qda_launch_quantize(x, rows, D, GS, bits, in_dt, packed, static_cast<uint16_t*>(scales),
                                      static_cast<uint16_t*>(biases), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return QDA_OK;
}

int qdecode_cache_append(const uint32_t* k_packed, const void* k_scales, const void* k_biases,
                         const uint32_t* v_packed, const void* v_scales, const void* v_biases, const float* k_new,
                         const float* v_new, uint32_t* k_packed_out, void* k_scales_out, void* k_biases_out,
                         uint32_t* v_packed_out, void* v_scales_out, void* v_biases_out, int B, int Hkv,
                         const int32_t* N, int T, int D, int GS, int bits, int dtype, void* stream) {
  if (!k_new || !v_new || !k_packed_out || !k_scales_out || !k_biases_out || !v_packed_out || !v_scales_out ||
      !v_biases_out || N == nullptr)
    return QDA_ERR_INVALID;
  if (B < 1 || Hkv < 1 || T < 1 || D < 1 || GS < 1) return QDA_ERR_INVALID;
  int in_dt, out_dt;
  int st = check_dtype(dtype, &in_dt, &out_dt);
  if (st != QDA_OK) return st;
  if (bits != 4 && bits != 8) return QDA_ERR_UNSUPPORTED;
  if (GS != 32 && GS != 64 && GS != 128) return QDA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256 && D != 512) return QDA_ERR_UNSUPPORTED;
  if (D % GS != 0 || B > QDA_MAX_B) return QDA_ERR_UNSUPPORTED;
  long long total_old = 0;
  for (int b = 0; b < B; ++b) {
    if (N[b] < 0) return QDA_ERR_INVALID;
    total_old += N[b];
  }
  if (total_old + (long long)B * T > (1LL << 31) - 1) return QDA_ERR_UNSUPPORTED;   // sequence offsets are int32
  if (total_old > 0 && (!k_packed || !k_scales || !k_biases || !v_packed || !v_scales || !v_biases))
    return QDA_ERR_INVALID;
  const void* ptrs[10] = {k_new, v_new, k_packed_out, k_scales_out, k_biases_out, v_packed_out, v_scales_out,
                          v_biases_out, k_packed, v_packed};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return QDA_ERR_ALIGN;
  QdaRowMap m;
  std::memset(&m, 0, sizeof(m));
  m.append = 1;
  m.B = B;
  m.Hkv = Hkv;
  m.T = T;
  for (int b = 0; b < B; ++b) {
    m.n_old[b] = N[b];
    m.off_old[b + 1] = m.off_old[b] + N[b];
    m.off_new[b + 1] = m.off_new[b] + N[b] + T;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int W = D * bits / 32, NG = D / GS;
  // the new rows' two quantizer launches first (an ordinary launch: it waits for whatever the stream did before),
  // then the old rows' copy; the second and third launches overlap their predecessors (they read nothing those
  // write) and each completes only after its predecessor, so the copy's completion ends the whole append
  const long long rows_new = (long long)B * Hkv * T;
  cudaError_t e = qda_launch_quantize(k_new, rows_new, D, GS, bits, in_dt, k_packed_out,
                                      static_cast<uint16_t*>(k_scales_out), static_cast<uint16_t*>(k_biases_out), s,
                                      &m, false);
  if (e != cudaSuccess) return cuda_fail(e);
  e = qda_launch_quantize(v_new, rows_new, D, GS, bits, in_dt, v_packed_out, static_cast<uint16_t*>(v_scales_out),
                          static_cast<uint16_t*>(v_biases_out), s, &m, true);
  if (e != cudaSuccess) return cuda_fail(e);
  e = qda_launch_append_copy(
      k_packed, static_cast<const uint16_t*>(k_scales), static_cast<const uint16_t*>(k_biases), v_packed,
      static_cast<const uint16_t*>(v_scales), static_cast<const uint16_t*>(v_biases), k_packed_out,
      static_cast<uint16_t*>(k_scales_out), static_cast<uint16_t*>(k_biases_out), v_packed_out,
      static_cast<uint16_t*>(v_scales_out), static_cast<uint16_t*>(v_biases_out), (long long)Hkv * total_old, W, NG,
      m, s, true);
  if (e != cudaSuccess) return cuda_fail(e);
  return QDA_OK;
}

const char* qdecode_attn_strerror(int status) {
  switch (status) {
    case QDA_OK: return "success";
    case QDA_ERR_INVALID: return "invalid argument (null pointer, non-positive size, H % Hkv != 0, N[b] < 1 or bad dtype)";
    case QDA_ERR_UNSUPPORTED: return "unsupported shape (bits, GS, D, B or H/Hkv outside the built variants)";
    case QDA_ERR_ALIGN: return "a data pointer is not 16-byte aligned";
    case QDA_ERR_CUDA: return "CUDA runtime error (see qdecode_attn_last_cuda_error)";
    case QDA_ERR_WORKSPACE: return "installed workspace is too small for this call";
    case QDA_ERR_SCRATCH: return "call needs more scratch than the fixed array of qdecode_attn_noalloc holds";
    default: return "unknown status";
  }
}

int qdecode_attn_last_cuda_error(void) { return t_last_cuda_error; }

int qdecode_attn_device_status(unsigned int* flags) {
  if (flags == nullptr) return QDA_ERR_INVALID;
  int dev;
  DeviceState* d = device_state(&dev);
  if (d == nullptr) return QDA_ERR_CUDA;
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_err, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e);
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_err, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = v;
  return QDA_OK;
}

long long qdecode_attn_calls(void) { return g_calls.load(); }

}  // extern "C"
