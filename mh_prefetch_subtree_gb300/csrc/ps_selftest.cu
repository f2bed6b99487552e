// Device-side check of the failure path that every bulk-copy wait of the
// scoring kernel takes: a bounded wait on an mbarrier that nothing completes
// gives up at its time limit and reports PS_DEV_TIMEOUT, and the context
// stays usable.  A diagnostic for tests; not a step of the method.
#include "ps_internal.cuh"

namespace ps {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t limit_ns, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        // no thread arrives and no copy signals this barrier, so its first
        // phase never completes: the wait ends by its limit
        if (!mbar_wait_bounded(&bar, 0, limit_ns)) set_status(status, PS_DEV_TIMEOUT);
    }
    __syncwarp();
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t *status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace ps
