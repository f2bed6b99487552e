// Round carry-over: the reached state's per-position values for the next
// round (PreSTO section 3.2 step (3): the sampler keeps the token-level log-
// probabilities of the state it moves to, for the next acceptance
// computations), with eq. (21) log-likelihood and eq. (22) confidence.
//
// One CTA per chain.  The reached state is x_{0:c*} + y^{s*} (Condition 1
// keeps every state in this form), so position t takes: the previous round's
// value if t <= the root's cut, else the root's row if t <= c*, else the row
// of s*.  The statistics are block reductions in a fixed order.
#include <math.h>

#include "ps_internal.cuh"

namespace ps {
namespace {

constexpr int kCarryThreads = 256;

__global__ void __launch_bounds__(kCarryThreads) carry_kernel(const CarryParams p) {
    __shared__ double red[2][kCarryThreads / 32];
    const int c = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const double qnan = __longlong_as_double(0x7ff8000000000000ll);
    const ps_carry_io &io = p.io;
    const int32_t T = p.T;
    const int64_t o = (int64_t)c * T;
    pdl_wait_prerequisites();              // the walk's state_seg is now visible

    const int32_t s0 = p.chain_seg0[c], s1 = p.chain_seg0[c + 1];
    bool ok = s0 >= 0 && s1 <= p.n_seg && s1 > s0;
    int32_t ss = 0, rc = 0, cstar = T;
    int64_t r0 = 0, y0 = 0;
    if (ok) {
        ss = io.state_seg[c];
        rc = p.seg_cut[s0];
        r0 = p.seg_row0[s0];
        ok = ss >= s0 && ss < s1 && rc >= 0 && rc <= T && p.seg_row0[s0 + 1] - r0 == T - rc &&
             p.seg_row0[s0 + 1] <= p.n_rows;
        if (ok && ss != s0) {
            cstar = p.seg_cut[ss];
            y0 = p.seg_row0[ss];
            ok = cstar >= 0 && cstar <= T - 1 && p.seg_row0[ss + 1] - y0 == T - cstar &&
                 p.seg_row0[ss + 1] <= p.n_rows;
        }
        if (ok && rc > 0 && (!io.prev_lp0 || !io.prev_lq)) ok = false;
        if (ok && rc > 0 && io.next_entropy && !io.prev_entropy) ok = false;
    }
    const bool ent = io.next_entropy != nullptr;
    double sl = 0.0, se = 0.0;
    for (int32_t t = 1 + tid; t <= T; t += kCarryThreads) {
        double v0 = qnan, vq = qnan, ve = qnan;
        if (ok) {
            if (t <= rc) {                              // carried from the previous round
                v0 = io.prev_lp0[o + t - 1];
                vq = io.prev_lq[o + t - 1];
                if (ent) ve = io.prev_entropy[o + t - 1];
            } else {
                const int64_t r = (t <= cstar) ? r0 + (t - rc - 1) : y0 + (t - cstar - 1);
                v0 = io.row_lp0[r];
                vq = io.row_lq[r];
                if (ent) ve = io.row_entropy[r];
            }
        }
        io.next_lp0[o + t - 1] = v0;
        io.next_lq[o + t - 1] = vq;
        if (ent) io.next_entropy[o + t - 1] = ve;
        sl += v0;
        se += ve;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        sl += __shfl_xor_sync(0xffffffffu, sl, off);
        se += __shfl_xor_sync(0xffffffffu, se, off);
    }
    if (lane == 0) {
        red[0][warp] = sl;
        red[1][warp] = se;
    }
    __syncthreads();
    if (tid == 0) {
        if (!ok) set_status(io.status, PS_DEV_BAD_LAYOUT);
        double a = 0.0, b = 0.0;
        for (int w = 0; w < kCarryThreads / 32; ++w) {
            a += red[0][w];
            b += red[1][w];
        }
        if (io.loglik) io.loglik[c] = ok ? a / T : qnan;
        if (io.confidence) io.confidence[c] = ok ? -b / T : qnan;
    }
}

}  // namespace

cudaError_t launch_carry(const CarryParams &p, cudaStream_t stream) {
    if (p.n_chains <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_chains);
    cfg.blockDim = dim3(kCarryThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, carry_kernel, p);
}

}  // namespace ps
