// K2: per-request suffix sums and log A (PreSTO eq. (6); Appendix B.1,
// eq. (7)-(9)).
//
// For request i with cut c_i and from-state segment src (chain root r0 with
// cut c_r):
//   y sum: the rows of segment i (positions c_i+1..T);
//   x sum: root rows for positions c_i+1..c_src, then all rows of src
//          (c_src = T and no src rows when src is the root).
// Condition 1 makes every state of the subtree x_{0:c_last} + y^last, which is
// why two contiguous row ranges hold the whole x suffix.
//   r_i = (LQ_x - LQ_y) + alpha (LP_y - LP_x),  log A_i = min{0, r_i}.
//
// One CTA per chain, one warp per request.  Each warp sums its ranges in
// float64 with lanes striding over rows and a fixed butterfly, so results are
// bit-reproducible.  Every index is checked before use; a failing request gets
// NaN outputs and a status bit.
#include <math.h>

#include "ps_internal.cuh"

namespace ps {
namespace {

constexpr int kAssembleThreads = 256;

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kAssembleThreads) assemble_kernel(const AssembleParams p) {
    const int c = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const double qnan = __longlong_as_double(0x7ff8000000000000ll);

    const int32_t s0 = p.chain_seg0[c];
    const int32_t s1 = p.chain_seg0[c + 1];
    if (s0 < 0 || s1 > p.n_seg || s1 <= s0) {
        if (threadIdx.x == 0) set_status(p.status, PS_DEV_BAD_LAYOUT);
        return;
    }
    const int32_t T = p.T;
    const int32_t rc = p.seg_cut[s0];
    const int64_t r0 = p.seg_row0[s0];
    const int64_t r1 = p.seg_row0[s0 + 1];
    const bool root_ok = p.seg_src[s0] == -1 && rc >= 0 && rc <= T && r0 >= 0 &&
                         r1 <= p.n_rows && r1 - r0 == (int64_t)(T - rc);

    if (threadIdx.x == 0) {
        if (!root_ok) set_status(p.status, PS_DEV_BAD_LAYOUT);
        double *outs[6] = {p.lp_y, p.lq_y, p.lp_x, p.lq_x, p.log_ratio, p.log_accept};
        for (int j = 0; j < 6; ++j)
            if (outs[j]) outs[j][s0] = qnan;
    }

    for (int32_t s = s0 + 1 + warp; s < s1; s += nwarps) {
        const int32_t cs = p.seg_cut[s];
        const int32_t src = p.seg_src[s];
        const int64_t y0 = p.seg_row0[s];
        const int64_t y1 = p.seg_row0[s + 1];
        int32_t bits = root_ok ? 0 : PS_DEV_BAD_LAYOUT;
        if (cs < 0 || cs > T - 1 || y0 < 0 || y1 > p.n_rows || y1 - y0 != (int64_t)(T - cs))
            bits |= PS_DEV_BAD_LAYOUT;
        if (src != s0 && (src <= s0 || src >= s1 || src == s)) bits |= PS_DEV_BAD_LAYOUT;
        int32_t csrc = T;
        int64_t q0 = 0, q1 = 0;
        if (bits == 0 && src != s0) {
            csrc = p.seg_cut[src];
            q0 = p.seg_row0[src];
            q1 = p.seg_row0[src + 1];
            if (csrc < 0 || csrc > T - 1 || q0 < 0 || q1 > p.n_rows ||
                q1 - q0 != (int64_t)(T - csrc))
                bits |= PS_DEV_BAD_LAYOUT;
        }
        if (bits == 0 && (cs > csrc || cs < rc)) bits |= PS_DEV_INFEASIBLE;

        double ly = qnan, qy = qnan, lx = qnan, qx = qnan;
        if (bits == 0) {
            double a = 0.0, b = 0.0;
            for (int64_t r = y0 + lane; r < y1; r += 32) {
                a += p.lp0[r];
                b += p.lq[r];
            }
            ly = warp_sum(a);
            qy = warp_sum(b);
            a = 0.0;
            b = 0.0;
            const int64_t x0 = r0 + (cs - rc), x1 = r0 + (csrc - rc);
            for (int64_t r = x0 + lane; r < x1; r += 32) {
                a += p.lp0[r];
                b += p.lq[r];
            }
            for (int64_t r = q0 + lane; r < q1; r += 32) {
                a += p.lp0[r];
                b += p.lq[r];
            }
            lx = warp_sum(a);
            qx = warp_sum(b);
        }
        if (lane == 0) {
            if (bits) set_status(p.status, bits);
            const double r = (qx - qy) + p.alpha * (ly - lx);
            const double la = (r != r) ? qnan : fmin(0.0, r);
            if (p.lp_y) p.lp_y[s] = ly;
            if (p.lq_y) p.lq_y[s] = qy;
            if (p.lp_x) p.lp_x[s] = lx;
            if (p.lq_x) p.lq_x[s] = qx;
            if (p.log_ratio) p.log_ratio[s] = r;
            p.log_accept[s] = la;
        }
    }
}

}  // namespace

cudaError_t launch_assemble(const AssembleParams &p, cudaStream_t stream) {
    if (p.n_chains <= 0) return cudaSuccess;
    assemble_kernel<<<p.n_chains, kAssembleThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ps
