// ptx.cuh -- inline-PTX helpers shared by the kernels that stage data through
// shared memory with mbarriers: barrier init/arrive/wait, bulk (TMA) copies
// and a bounded wait.
#pragma once

#include <stdint.h>

namespace moe {

constexpr unsigned long long kTimeoutNs = 2000000000ull;   // bounded waits give up after ~2 s
constexpr uint32_t kWaitSliceNs = 20000;                    // longest park per try_wait

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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
// try_wait with a suspend-time hint: a thread whose phase is not complete is
// parked (it issues nothing) until the phase completes or about `ns`
// nanoseconds pass, instead of spinning and taking issue slots from the warps
// that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// Arrive on the barrier at the same shared-memory offset in CTA `rank` of the
// cluster, with the default (CTA-scope) release: the arrival orders nothing
// but the thread's own shared-memory and tensor-memory work that the caller
// has already completed and fenced, so it does not wait for the thread's
// outstanding global stores the way a cluster-scope release does.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t *bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync, for a barrier whose wait can come later
// than the arrive (work in between overlaps the slower CTAs).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One-dimensional bulk copy global -> shared, completing on `bar` (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 eviction-priority policies (cache hints for stores and bulk copies): a
// line stored with evict_last is kept over normal and evict_first lines.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// bulk_load with an L2 cache policy for the global reads.
__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes,
                                               uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Waits for phase `parity` of `bar`.  Gives up when the CTA's abort flag is set
// or after limit_ns (kTimeoutNs unless a caller passes a shorter limit),
// setting the abort flag and the status bit.  The first test is inline; the
// bounded loop is a separate function entered only when the phase is not
// complete yet, so that a wait which succeeds at once costs one instruction
// and no call (a call spills the caller's live registers).
static __device__ __noinline__ bool wait_bounded_loop(uint64_t *bar, uint32_t parity,
                                                      volatile int *abort_flag, int32_t *status,
                                                      bool honour_abort,
                                                      unsigned long long limit_ns = kTimeoutNs) {
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSliceNs)) return true;
        if (honour_abort && *abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            if (status) atomicOr(status, MOE_DEV_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                             int32_t *status, bool honour_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bounded_loop(bar, parity, abort_flag, status, honour_abort);
}
}  // namespace moe
