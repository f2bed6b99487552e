// Diagnostics for tests and measurement; not steps of the method.
//
// wait_selftest_kernel: the failure path that every bulk-copy wait of the
// scoring kernel takes: a bounded wait on an mbarrier that nothing completes
// gives up at its time limit and reports PS_DEV_TIMEOUT, and the context
// stays usable.
//
// read_probe_kernel: a plain streaming read of a device buffer, the rate the
// scoring kernel's own read rate is compared with.  16-byte streaming loads,
// eight in flight per thread, four 512-thread blocks per SM striding through
// the buffer; the words are combined with XOR and each warp folds its value
// into one output word, so that no load can be dropped.
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

constexpr int kProbeThreads = 512;
constexpr int kProbeBlocksPerSm = 4;
constexpr int kProbeInFlight = 8;

__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4 *p, int64_t n_vec,
                                                                    uint32_t *sink) {
    const int64_t stride = (int64_t)gridDim.x * kProbeThreads;
    int64_t i = (int64_t)blockIdx.x * kProbeThreads + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (kProbeInFlight - 1) * stride < n_vec; i += kProbeInFlight * stride) {
        uint4 v[kProbeInFlight];
#pragma unroll
        for (int j = 0; j < kProbeInFlight; ++j) v[j] = __ldcs(p + i + j * stride);
#pragma unroll
        for (int j = 0; j < kProbeInFlight; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
    }
    for (; i < n_vec; i += stride) {
        const uint4 v = __ldcs(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace

cudaError_t launch_read_probe(const void *data, int64_t n_vec, uint32_t *sink, int sms,
                              cudaStream_t stream) {
    if (n_vec <= 0) return cudaSuccess;
    read_probe_kernel<<<sms * kProbeBlocksPerSm, kProbeThreads, 0, stream>>>(
        static_cast<const uint4 *>(data), n_vec, sink);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t *status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace ps
