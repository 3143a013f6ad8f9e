// tma.cuh -- bulk asynchronous copies (TMA, 1-D) and mbarriers, inline PTX.
//
// Every wait is bounded: after the caller's limit (kWaitNs unless a test
// shortens it) or kWaitLimit polls the waiter gives up and reports false, so
// a copy that never lands cannot hang the GPU; the caller then marks its
// results invalid and reports the timeout in the device status word.  A waiting thread is
// suspended by the hardware between polls, so waiters take no issue slots
// from the warps that still work.
#pragma once

#include <stdint.h>

namespace spf {

constexpr uint32_t kWaitLimit = 1u << 22;       // polls
constexpr uint64_t kWaitNs = 2000000000ull;      // 2 s
constexpr uint32_t kSuspendNs = 100000;          // longest suspension per poll

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make the barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}

// As mbar_try_wait, letting the hardware suspend the thread for up to `ns`
// nanoseconds while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0u;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; false after
// `limit_ns` nanoseconds (or kWaitLimit polls) without it.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  // the clock is read once per 64 polls (and on the first one): %globaltimer
  // read in a tight loop on many SMs slows every reader of it
  const uint64_t t0 = global_ns();
  const uint32_t suspend = limit_ns < kSuspendNs ? (uint32_t)limit_ns : kSuspendNs;
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait_suspend(bar, parity, suspend)) return true;
    if ((i & 63u) == 0u && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned) completing on `bar`, with an evict-first L2 policy
// (the data is read once).
__device__ __forceinline__ void tma_load_1d(void* dst_smem, const void* src, uint32_t bytes,
                                           uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Start bringing `bytes` (a multiple of 16) of global memory at a 16-byte
// aligned address into L2, without waiting.  A hint only: a later load of
// the same bytes reads what is current, so it may go out before the kernel
// that writes them has finished (L2 is the device's point of coherence).
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

}  // namespace spf
