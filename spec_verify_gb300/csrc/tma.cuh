// Bulk (1-D) TMA copies into shared memory with mbarrier completion, and the
// bounded wait on them, shared by the streaming kernels.
#pragma once

#include "common.cuh"

namespace smp {

// L2 policy for data read once: evicted before anything else, so that a row
// streaming through L2 does not push out the kernel's code and small inputs.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// One bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// into shared memory, completing on `bar`; bytes == 0 only arrives on it.
__device__ __forceinline__ void tma_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
  if (bytes)
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// The same without an L2 policy (data that is read again soon).
__device__ __forceinline__ void tma_load_keep(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
  if (bytes)
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// L2 prefetch of [src, src + bytes) (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(uintptr_t src, uint32_t bytes) {
  if (bytes) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Wait (every thread) for a TMA phase; false after `limit_ns`.  A limit of
// 0 tests the phase once without waiting (mbarrier.try_wait may suspend the
// thread until the phase completes, so it is not used for that test).
__device__ __forceinline__ bool wait_full(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (limit_ns == 0) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
  }
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 255u) == 255u && global_timer_ns() - t0 > limit_ns) return false;
  }
}

}  // namespace smp
