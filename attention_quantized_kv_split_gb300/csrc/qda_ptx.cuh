// Inline-PTX helpers for sm_103a: mbarriers, 1-D bulk copies (TMA), programmatic dependent launch, timers.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace qda {

// Index checks of a checked build (compiled with QDA_BOUNDS_CHECK): a failed check sets bit 4 of the device error
// word and the caller skips the access. In the normal build every check is the constant true.
#ifdef QDA_BOUNDS_CHECK
__device__ __forceinline__ bool in_bounds(bool ok, unsigned int* err) {
  if (!ok) atomicOr(err, 4u);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, unsigned int*) { return true; }
#endif

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy before any copy signals it.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` inside the call while the phase is incomplete (it
// wakes when the phase completes), so a waiting warp does not spend issue slots polling.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on a barrier phase. Gives up after `limit_ns` (or as soon as *abort is set by another thread),
// records `code` in the device error word and raises *abort; returns whether the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  unsigned int* err, unsigned int code,
                                                  uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, code);
      *abort = 1;
      return false;
    }
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of transaction count on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once (the cache stream): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: let the dependent grid start its prologue / wait for the primary grid.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float bf16_bits_to_float(uint32_t u16) { return __uint_as_float(u16 << 16); }

__device__ __forceinline__ float fp16_bits_to_float(uint32_t u16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(u16)));
}

template <bool F16>
__device__ __forceinline__ float half_bits_to_float(uint32_t u16) {
  if constexpr (F16) {
    return fp16_bits_to_float(u16);
  } else {
    return bf16_bits_to_float(u16);
  }
}

// bf16 or fp16 bits -> float, dtype chosen at run time (a warp-uniform select)
__device__ __forceinline__ float half_bits_to_float_rt(uint32_t u16, bool f16) {
  return f16 ? fp16_bits_to_float(u16) : bf16_bits_to_float(u16);
}

// Two bf16 or fp16 values packed in a word (first in the low half) -> float2, dtype chosen at run time.
__device__ __forceinline__ float2 half2_bits_to_float2_rt(uint32_t w, bool f16) {
  if (f16) return __half22float2(*reinterpret_cast<const __half2*>(&w));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

}  // namespace qda
