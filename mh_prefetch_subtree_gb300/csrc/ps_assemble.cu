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
//   r_i = (LQ_x - LQ_y) + alpha (LP_y - LP_x),  log A_i = min{0, r_i},
// and, when asked, the epsilon-certainty class of the decision (section 3.3).
//
// One CTA per segment (a chain root only writes NaN to its own entries).  It
// is launched with programmatic dependent launch, so its CTAs may start while
// the previous kernel finishes; griddepcontrol.wait makes all of that
// kernel's writes visible before they are read.  The threads stride over the
// rows in float64 and the block reduces in a fixed order (warp butterfly, then
// warps in index order), so results are bit-reproducible.  Every index is
// checked before use; a failing request gets NaN outputs and a status bit.
//
// The fused form, used when one call scores, sums and walks, also takes the
// walk (section 3.2 step (3)): the last CTA of each chain to write its log A
// walks the chain, so the round needs no third launch.
#include <math.h>

#include <type_traits>

#include "ps_walk_chain.cuh"

namespace ps {
namespace {

// 256 threads per segment: wider blocks measured slower (1024 threads took
// 17 us instead of 11 on the long-context batch), since they hold fewer loads
// in flight per thread and wait longer at the block reduction.
constexpr int kAssembleThreads = 256;

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// A request's sums over four row ranges laid end to end in one index space:
// range 0 (the y rows) goes to (a, b), ranges 1-3 (the x suffix) to (e, f).
// Range k reads lp_k[o_k + j], lq_k[o_k + j] for j < n_k.  The threads stride
// over the index space and issue the loads of up to kU indices before adding
// any (2,048 indices per round for the block), so a request's sums usually
// take one or two rounds of memory latency.  Each thread adds its elements in
// index order: the result is deterministic.  (Deeper rounds, 12 or 16 loads
// per thread, measured slower: they take more registers per thread.)
struct Ranges {
    const double *lp[4];
    const double *lq[4];
    int64_t o[4];
    int64_t n[4];
};

__device__ __forceinline__ void ranges_sum(const Ranges &g, int tid, double &a, double &b,
                                           double &e, double &f) {
    constexpr int kU = 8;
    const int64_t e0 = g.n[0], e1 = e0 + g.n[1], e2 = e1 + g.n[2], e3 = e2 + g.n[3];
    for (int64_t base = tid; base < e3; base += (int64_t)kU * kAssembleThreads) {
        double x[kU], y[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            const int64_t i = base + (int64_t)j * kAssembleThreads;
            x[j] = y[j] = 0.0;
            if (i < e3) {
                const bool r0 = i < e0, r1 = i < e1, r2 = i < e2;
                const int64_t off = r0 ? g.o[0] + i
                                       : (r1 ? g.o[1] + (i - e0)
                                             : (r2 ? g.o[2] + (i - e1) : g.o[3] + (i - e2)));
                const double *pl = r0 ? g.lp[0] : (r1 ? g.lp[1] : (r2 ? g.lp[2] : g.lp[3]));
                const double *pq = r0 ? g.lq[0] : (r1 ? g.lq[1] : (r2 ? g.lq[2] : g.lq[3]));
                x[j] = __ldcg(pl + off);
                y[j] = __ldcg(pq + off);
            }
        }
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            const int64_t i = base + (int64_t)j * kAssembleThreads;
            if (i < e0) {
                a += x[j];
                b += y[j];
            } else if (i < e3) {
                e += x[j];
                f += y[j];
            }
        }
    }
}

// Adds 1 to *cnt with release and acquire semantics at GPU scope and returns
// the old value: the caller's earlier writes are visible to whichever thread
// later sees the sum, and the writes of the threads whose additions came
// before are visible to the caller.
__device__ __forceinline__ int32_t arrive_acq_rel(int32_t *cnt) {
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(cnt)
                 : "memory");
    return old;
}

// Chain holding segment s: the last c with chain_seg0[c] <= s.
__device__ int chain_of(const int32_t *chain_seg0, int n_chains, int32_t s) {
    int lo = 0, hi = n_chains - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chain_seg0[mid] <= s) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// One block per segment.  FUSED: the last CTA of each
// chain to finish (arrivals counted in chain_cnt, zeroed before the launch)
// also walks that chain with its first warp, so that the walk needs no launch
// of its own.  EARLY: the kernel directly follows libps's own scoring kernel,
// launched in the same call, so the caller's inputs were written before that
// kernel started and the metadata may be loaded before griddepcontrol.wait
// (with FUSED, every CTA's first warp also stages its chain's tree and
// uniforms then, in case it is the one that walks); only the per-row values
// wait.  Without EARLY nothing is read before the wait, because the previous
// kernel may be the caller's own kernel writing the layout arrays.
//
// The early fused form holds its chain's bounds through the sums; its bound of
// three CTAs per SM keeps it at the occupancy of the others (at most 85
// registers a thread), which matters when a batch has thousands of segments.
template <bool FUSED, bool EARLY>
__global__ void __launch_bounds__(kAssembleThreads, (FUSED && EARLY) ? 3 : 0)
    assemble_kernel(const AssembleParams p, const WalkParams wp, int32_t *chain_cnt) {
    constexpr int kWarps = kAssembleThreads / 32;
    __shared__ double red[4][kWarps];
    __shared__ typename std::conditional<FUSED, WalkSmem, int>::type wsm;
    __shared__ int walk_here;
    const int32_t s = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const double qnan = __longlong_as_double(0x7ff8000000000000ll);
    pdl_launch_dependents();                         // the next kernel may be scheduled now
    if constexpr (!EARLY) pdl_wait_prerequisites();
    const int c = chain_of(p.chain_seg0, p.n_chains, s);
    ChainStage stage{};
    if constexpr (FUSED && EARLY) {
        if (warp == 0) stage = stage_chain(wp, c, wsm, lane);
    }
    // metadata in two rounds of loads: what depends on s (and c) only, then
    // the root's and src's entries (indices clamped in range, checked below)
    const int32_t s0 = p.chain_seg0[c];
    const int32_t s1 = p.chain_seg0[c + 1];
    const int32_t cs = p.seg_cut[s];
    const int32_t src = p.seg_src[s];
    const int64_t y0 = p.seg_row0[s];
    const int64_t y1 = p.seg_row0[s + 1];
    const bool chain_ok = s0 >= 0 && s1 <= p.n_seg && s1 > s0 && s >= s0 && s < s1;
    const bool root = chain_ok && s == s0;           // a chain root: NaN entries only
    const int32_t T = p.T;
    int32_t bits = chain_ok ? 0 : PS_DEV_BAD_LAYOUT;
    double ly = qnan, qy = qnan, lx = qnan, qx = qnan;
    if (!root) {
        const int32_t s0l = bits ? s : s0;
        const bool src_root = src == s0;
        const bool src_ok = src_root || (src > s0 && src < s1 && src != s);
        const int32_t srcl = (bits == 0 && src_ok) ? src : s;
        const int32_t rc = p.seg_cut[s0l];
        const int32_t rsrc = p.seg_src[s0l];
        const int64_t r0 = p.seg_row0[s0l];
        const int64_t r1 = p.seg_row0[s0l + 1];
        const int32_t csrc_l = p.seg_cut[srcl];
        const int64_t q0_l = p.seg_row0[srcl];
        const int64_t q1_l = p.seg_row0[srcl + 1];
        if (bits == 0) {
            if (rsrc != -1 || rc < 0 || rc > T || r0 < 0 || r1 > p.n_rows ||
                r1 - r0 != (int64_t)(T - rc))
                bits |= PS_DEV_BAD_LAYOUT;
            if (cs < 0 || cs > T - 1 || y0 < 0 || y1 > p.n_rows || y1 - y0 != (int64_t)(T - cs))
                bits |= PS_DEV_BAD_LAYOUT;
            if (!src_ok) bits |= PS_DEV_BAD_LAYOUT;
        }
        int32_t csrc = T;
        int64_t q0 = 0, q1 = 0;
        if (bits == 0 && !src_root) {
            csrc = csrc_l;
            q0 = q0_l;
            q1 = q1_l;
            if (csrc < 0 || csrc > T - 1 || q0 < 0 || q1 > p.n_rows ||
                q1 - q0 != (int64_t)(T - csrc))
                bits |= PS_DEV_BAD_LAYOUT;
        }
        // Condition 1; and without carried root values, the root rows must
        // cover every position a request's x suffix reads
        if (bits == 0 && (cs > csrc || (cs < rc && p.root_lp0 == nullptr)))
            bits |= PS_DEV_INFEASIBLE;

        if constexpr (EARLY) pdl_wait_prerequisites();   // per-row values are now visible
        if (bits == 0) {                                 // uniform across the block
            double a = 0.0, b = 0.0, e = 0.0, f = 0.0;
            // y: the request's own rows.  x: positions cs+1..csrc of the current
            // state (carried values up to the root's cut, root rows above it),
            // then all rows of src
            const int32_t k1 = min(rc, csrc);               // last carried position
            const int32_t lo = max(cs, rc);                 // rows cover positions > rc
            Ranges g;
            g.lp[0] = p.lp0, g.lq[0] = p.lq, g.o[0] = y0, g.n[0] = y1 - y0;
            g.lp[1] = p.root_lp0, g.lq[1] = p.root_lq, g.o[1] = (int64_t)c * T + cs;
            g.n[1] = cs < k1 ? (int64_t)(k1 - cs) : 0;
            g.lp[2] = p.lp0, g.lq[2] = p.lq, g.o[2] = r0 + (lo - rc);
            g.n[2] = lo < csrc ? (int64_t)(csrc - lo) : 0;
            g.lp[3] = p.lp0, g.lq[3] = p.lq, g.o[3] = q0, g.n[3] = q1 - q0;
            ranges_sum(g, tid, a, b, e, f);
            a = warp_sum(a);
            b = warp_sum(b);
            e = warp_sum(e);
            f = warp_sum(f);
            if (lane == 0) {
                red[0][warp] = a;
                red[1][warp] = b;
                red[2][warp] = e;
                red[3][warp] = f;
            }
            __syncthreads();
            if (tid == 0) {
                ly = qy = lx = qx = 0.0;
                for (int w = 0; w < kWarps; ++w) {
                    ly += red[0][w];
                    qy += red[1][w];
                    lx += red[2][w];
                    qx += red[3][w];
                }
            }
        }
    }
    // a chain root reads no per-row value, but it waits as well, so that no CTA
    // of this kernel ends before the scoring kernel has
    if constexpr (EARLY) {
        if (root) pdl_wait_prerequisites();
    }
    if (tid == 0) {
        if (bits) set_status(p.status, bits);
        if (root) {
            double *outs[6] = {p.lp_y, p.lq_y, p.lp_x, p.lq_x, p.log_ratio, p.log_accept};
            for (int j = 0; j < 6; ++j)
                if (outs[j]) outs[j][s] = qnan;
            if (p.eps_class) p.eps_class[s] = -1;
        } else {
            const double r = (qx - qy) + p.alpha * (ly - lx);
            const double la = (r != r) ? qnan : fmin(0.0, r);
            if (p.lp_y) p.lp_y[s] = ly;
            if (p.lq_y) p.lq_y[s] = qy;
            if (p.lp_x) p.lp_x[s] = lx;
            if (p.lq_x) p.lq_x[s] = qx;
            if (p.log_ratio) p.log_ratio[s] = r;
            p.log_accept[s] = la;
            if (p.eps_class) {
                // epsilon-certainty (section 3.3), compared in the log domain:
                // A <= eps  <=>  log A <= log eps;  A >= 1 - eps  <=>  log A >= log1p(-eps)
                int8_t cls = -1;
                if (la == la) cls = la <= log(p.eps) ? 0 : (la >= log1p(-p.eps) ? 2 : 1);
                p.eps_class[s] = cls;
            }
        }
    }
    if constexpr (FUSED) {
        // the last CTA of the chain to get here walks it (a chain whose
        // chain_seg0 bounds failed the checks above is not counted, so not
        // walked; its status bit is set).  Thread 0 wrote this CTA's outputs:
        // its release publishes them, and the last arrival's acquire, passed
        // on by the barrier, makes every arrival's log A visible to the warp
        // that walks.
        if (tid == 0)
            walk_here = chain_ok && arrive_acq_rel(chain_cnt + c) == s1 - s0 - 1;
        __syncthreads();
        if (walk_here && warp == 0) {
            if constexpr (!EARLY) stage = stage_chain(wp, c, wsm, lane);
            walk_staged(wp, c, stage, wsm, lane);
        }
    }
}

template <bool FUSED, bool EARLY>
cudaError_t launch_t(const AssembleParams &p, const WalkParams &wp, int32_t *chain_cnt,
                     cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_seg);
    cfg.blockDim = dim3(kAssembleThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, assemble_kernel<FUSED, EARLY>, p, wp, chain_cnt);
}

}  // namespace

cudaError_t launch_assemble(const AssembleParams &p, cudaStream_t stream) {
    if (p.n_seg <= 0 || p.n_chains <= 0) return cudaSuccess;
    const WalkParams none{};
    return launch_t<false, false>(p, none, nullptr, stream);
}

cudaError_t launch_assemble_walk(const AssembleParams &p, const WalkParams &wp,
                                 int32_t *chain_cnt, bool early, cudaStream_t stream) {
    if (p.n_seg <= 0 || p.n_chains <= 0) return cudaSuccess;
    return early ? launch_t<true, true>(p, wp, chain_cnt, stream)
                 : launch_t<true, false>(p, wp, chain_cnt, stream);
}

}  // namespace ps
