// selftest.cu -- moe_wait_selftest: the give-up path of the bounded waits.
//
// Every wait of the staged kernels (on a stage, accumulator or drain barrier)
// runs through wait_bounded_loop, which gives up after a time limit, sets
// MOE_DEV_TIMEOUT in the call's status word and lets the kernel leave.  In
// those kernels a wait only runs out if a copy or an MMA never completes, so
// the self-test exercises the same loop on a barrier that nothing arrives on,
// with no copy and no MMA attached: one thread waits on it with a
// caller-chosen short limit and must come back with the status bit set.
#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// status[0]: the status word; status[2..3]: nanoseconds the wait took.
__global__ void k_wait_selftest(int32_t *status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    pdl_wait();
    if (threadIdx.x != 0) return;
    *status = 0;
    abort_flag = 0;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint64_t t0 = globaltimer();
    // nothing arrives on `bar`: the first test fails and the bounded loop runs
    // until limit_ns have passed, then records MOE_DEV_TIMEOUT and returns
    if (!mbar_try_wait(&bar, 0))
        wait_bounded_loop(&bar, 0, &abort_flag, status, true, limit_ns);
    const uint64_t t1 = globaltimer();
    *reinterpret_cast<unsigned long long *>(status + 2) = t1 - t0;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_wait_selftest(void *workspace, size_t workspace_bytes, uint64_t limit_ns,
                             cudaStream_t stream) {
    if (!workspace) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (((uintptr_t)workspace % kAlign) != 0) return MOE_FAIL(MOE_ERR_ALIGNMENT);
    if (workspace_bytes < 16) return MOE_FAIL(MOE_ERR_WORKSPACE);
    if (limit_ns == 0 || limit_ns > kTimeoutNs) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    MOE_LAUNCH("wait_selftest", k_wait_selftest, 1, 32, 0, stream,
               static_cast<int32_t *>(workspace), (unsigned long long)limit_ns);
    return MOE_OK;
}

}  // extern "C"
