// ptx.cuh -- the mbarrier / TMA / elect glue shared by the persistent kernels
// (tensor-core grouped GEMM, TMA-fed GEMV).  Every wait is bounded by
// %globaltimer: a wait that gives up sets the device status word and the CTA's
// abort flag, and returns false so the caller can drain and exit.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "moe_internal.cuh"

namespace moe {

constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s per wait

static __device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

static __device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

static __device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

static __device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

static __device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The non-blocking test (try_wait may hold the thread for a while before it
// reports an incomplete phase; test_wait answers at once).
static __device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test, letting the thread sleep until the phase completes (or
// kSuspendNs passes): a polling warp then takes no issue slots from the
// warps that share its scheduler.
constexpr uint32_t kSuspendNs = 20000;
static __device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

static __device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: false if the CTA is stopping (*abort set) or the wait ran
// past kWaitNs (then *status and *abort are set).  The first test is
// inlined; only a wait that has to poll calls the out-of-line loop, which
// sleeps in the mbarrier between polls.
static __device__ __noinline__ bool wait_bar_slow(uint64_t *bar, uint32_t parity, int *abort,
                                                  int32_t *status) {
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*reinterpret_cast<volatile int *>(abort)) return false;
      if (globaltimer() - t0 > kWaitNs) {
        atomicExch(abort, 1);
        atomicExch(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Called by a whole warp.  Its lanes decide alike: they test the barrier
// together, and the phase cannot move on while they wait (the warp that
// releases it next is held by this warp's own next __syncwarp), so under a
// 2 s limit no lane can give up where another saw completion.
static __device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int *abort,
                                                int32_t *status) {
  return mbar_try_wait(bar, parity) || wait_bar_slow(bar, parity, abort, status);
}

// The same wait under a limit shorter than the default, for the kernels'
// short-wait instantiations (the limit test in the hot wait costs time, so
// the ordinary kernels never carry it): non-blocking tests -- try_wait may
// hold a thread past a short limit -- with the clock read after every one.
// A limit of 0 gives up at the first incomplete test.
static __device__ __noinline__ bool wait_bar_short_loop(uint64_t *bar, uint32_t parity, int *abort,
                                                        int32_t *status,
                                                        unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int *>(abort)) return false;
    if (globaltimer() - t0 >= limit_ns) {
      atomicExch(abort, 1);
      atomicExch(status, kStatusTimeout);
      return false;
    }
  }
}

// The role wait of a kernel instantiated with or without short waits.  Under
// a short limit a lane may give up within nanoseconds of another seeing the
// phase complete, so there the warp votes: every lane gets the same answer
// and the warp-collective instructions that follow (elect.sync, tcgen05.ld /
// st) are never reached by part of a warp.
template <bool kShortWaits>
static __device__ __forceinline__ bool wait_role(uint64_t *bar, uint32_t parity, int *abort,
                                                 int32_t *status, unsigned long long limit_ns) {
  if constexpr (kShortWaits)
    return __all_sync(0xffffffffu, wait_bar_short_loop(bar, parity, abort, status, limit_ns));
  else
    return wait_bar(bar, parity, abort, status);
}

// Spins (bounded) until the phase of `parity` completes; for draining copies
// before a CTA exits.
static __device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity,
                                                 unsigned long long t0) {
  while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < kWaitNs) {
  }
}

// Orders this thread's generic-proxy accesses to shared memory before later
// async-proxy (TMA, tcgen05) accesses once an mbarrier hands the buffer over.
// A stage that threads read with ordinary loads and then release for a TMA
// refill needs it: without it the refill can overwrite data still being read.
static __device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

static __device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                                   uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// An L2 policy that evicts the lines it covers first: for data read once
// (decode weights), so it does not push the workspace out of L2.
static __device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tma_load_2d with an L2 cache policy.
static __device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int x,
                                                        int y, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// One lane of a converged warp (elect.sync); role loops run warp-wide so
// coordinates and barrier addresses stay warp-uniform.
static __device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

}  // namespace moe
