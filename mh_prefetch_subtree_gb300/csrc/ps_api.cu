// Host side of libps: argument checks, workspace layout, launches, and the
// synchronous structural validator.  See include/ps.h for the contract.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "ps_internal.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: per-row values (when the caller does not ask for them), the
// split-row partials, then the per-chain arrival counters of the fused
// suffix-sum + walk kernel directly followed by the row kernel's arrival
// counters, so that one memset clears both.
struct WsLayout {
    size_t rows_off, rows_bytes;
    size_t parts_off, parts_bytes;
    size_t chain_cnt_off, chain_cnt_bytes;
    size_t cnt_off, cnt_bytes;
    size_t total;
};

WsLayout ws_layout(int64_t n_rows, int32_t n_chains) {
    WsLayout w;
    w.rows_off = 0;
    w.rows_bytes = align_up((size_t)(n_rows > 0 ? n_rows : 0) * 2 * sizeof(double), kAlign);
    w.parts_off = w.rows_off + w.rows_bytes;
    w.parts_bytes = align_up((size_t)2 * ps::kMaxRanges * sizeof(ps::RowPart), kAlign);
    w.chain_cnt_off = w.parts_off + w.parts_bytes;
    w.chain_cnt_bytes = align_up((size_t)(n_chains > 0 ? n_chains : 0) * sizeof(int32_t), kAlign);
    w.cnt_off = w.chain_cnt_off + w.chain_cnt_bytes;
    w.cnt_bytes = align_up((size_t)ps::kMaxRanges * sizeof(int32_t), kAlign);
    w.total = w.cnt_off + w.cnt_bytes;
    return w;
}

int elem_size(int32_t dtype) { return dtype == PS_BF16 ? 2 : (dtype == PS_F32 ? 4 : 0); }

// Device that owns `ptr`, made current for this thread; SM count cached.
ps_status device_of(const void *ptr, int *sms) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
        cudaGetLastError();
        return PS_ERR_INVALID_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return PS_ERR_INVALID_ARG;
    const int dev = attr.device;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return PS_ERR_CUDA;
    if (cur != dev && cudaSetDevice(dev) != cudaSuccess) return PS_ERR_CUDA;
    static std::mutex mu;
    static std::vector<int> cache;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PS_ERR_CUDA;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major * 10 + minor != 103) return PS_ERR_UNSUPPORTED;   // built for sm_103a only
        // the scoring kernel's rings need this much shared memory per CTA
        int smem = 0;
        if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            (size_t)smem < ps::score_rows_smem_bytes())
            return PS_ERR_UNSUPPORTED;
        cache[dev] = n;
    }
    *sms = cache[dev];
    return PS_OK;
}

ps_status map_cuda(cudaError_t e) { return e == cudaSuccess ? PS_OK : PS_ERR_CUDA; }

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// 1/tau when it is exactly 1, 2, 4 or 8 (then the tau exponential is a power).
int32_t integer_power(double tau) {
    const double g = 1.0 / tau;
    for (int n : {1, 2, 4, 8})
        if (g == (double)n) return n;
    return 0;
}

ps_status check_batch_host(const ps_subtree_batch *b, bool need_data = true) {
    if (!b) return PS_ERR_INVALID_ARG;
    if (b->V < 1 || b->T < 1 || b->n_chains < 1 || b->n_seg < b->n_chains || b->n_rows < 0)
        return PS_ERR_INVALID_ARG;
    if (b->flags & ~PS_FLAG_MASKED_LOGITS) return PS_ERR_INVALID_ARG;
    const int esz = elem_size(b->dtype);
    if (esz == 0) return PS_ERR_UNSUPPORTED;
    if (!(b->tau > 0.0) || !isfinite(b->tau) || !isfinite(b->alpha)) return PS_ERR_INVALID_ARG;
    const int64_t row_bytes = ((int64_t)b->V * esz + 15) / 16 * 16;
    if (row_bytes > (int64_t(1) << 30)) return PS_ERR_INVALID_ARG;   // chunk offsets are 32-bit
    if (b->ld < b->V || (b->ld * esz) % 16 != 0 || b->ld * esz < row_bytes)
        return PS_ERR_INVALID_ARG;
    if (!b->chain_seg0 || !b->seg_row0 || !b->seg_cut || !b->seg_src) return PS_ERR_INVALID_ARG;
    if (b->n_rows > 0 && need_data) {
        if (!b->logits || !b->tokens || !aligned(b->logits, 16)) return PS_ERR_INVALID_ARG;
        if (b->row_index) {
            if (b->n_logit_rows < 1) return PS_ERR_INVALID_ARG;
        } else if (b->n_logit_rows < b->n_rows) {
            return PS_ERR_INVALID_ARG;
        }
    }
    return PS_OK;
}

}  // namespace

extern "C" {

const char *ps_version(void) { return "libps 0.4.0 (sm_103a)"; }

const char *ps_status_string(ps_status s) {
    switch (s) {
        case PS_OK: return "ok";
        case PS_ERR_INVALID_ARG: return "invalid argument";
        case PS_ERR_INFEASIBLE: return "request violates Condition 1 (c_i > c_src)";
        case PS_ERR_BAD_TREE: return "inconsistent tree";
        case PS_ERR_UNSUPPORTED: return "unsupported dtype or device";
        case PS_ERR_CUDA: return "CUDA runtime error";
        case PS_ERR_TIMEOUT: return "device wait timed out";
        case PS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    }
    return "unknown status";
}

size_t ps_score_workspace_bytes(const ps_subtree_batch *batch) {
    if (!batch) return 0;
    return ws_layout(batch->n_rows, batch->n_chains).total;
}

}  // extern "C"

namespace {

// Where the row kernel keeps its scratch: the split-row partials, the arrival
// counters, and how many chunk ranges (one partial pair and one counter each)
// fit; one counter slot goes to the tail-block claim counter.  The memset
// before the launch clears [zero_from, the claim counter], so that counters
// placed just before the row kernel's are cleared with them.
struct RowsScratch {
    ps::RowPart *parts;
    int32_t *counters;
    int64_t max_ranges;
    int32_t *zero_from;
};

// Launch of the row kernel shared by every scoring entry point.  npow/g select
// the tau path; for the multi-temperature mode (npow == 16 or 17)
// tau_pow/n_taus/lq_multi replace lq.  The batch has been checked by
// check_batch_host and has at least one row.
ps_status launch_rows(const ps_subtree_batch *b, int sms, const RowsScratch &scr, double *lp0,
                      double *lq, double *entropy, int32_t *status, void *cuda_stream,
                      int32_t npow, float g, const int32_t *tau_pow, int32_t n_taus,
                      double *lq_multi) {
    cudaStream_t stream = (cudaStream_t)cuda_stream;
    const int esz = elem_size(b->dtype);
    ps::RowsParams p{};
    p.logits = (const uint8_t *)b->logits;
    p.ld_bytes = b->ld * esz;
    p.n_logit_rows = b->row_index ? b->n_logit_rows : b->n_rows;
    p.row_index = b->row_index;
    p.tokens = b->tokens;
    p.n_rows = b->n_rows;
    p.V = b->V;
    p.dtype = b->dtype;
    p.flags = b->flags;
    p.row_bytes = (int32_t)(((int64_t)b->V * esz + 15) / 16 * 16);
    p.cpr = (p.row_bytes + ps::kStageBytes - 1) / ps::kStageBytes;
    p.n_chunks = b->n_rows * p.cpr;
    int64_t warps = (int64_t)sms * ps::kWarpsPerCta;
    if (warps > scr.max_ranges - 1) warps = scr.max_ranges - 1;
    if (warps > p.n_chunks) warps = p.n_chunks;
    p.n_vwarps = (int32_t)warps;
    // On batches where each warp streams at least kTailMinShare chunks, static
    // ranges cover the first 15/16 of the chunks and the last 1/16 is cut
    // into tail blocks (up to 8 per warp, as the scratch allows, of at least
    // kTailMinBlock chunks) that the warps finishing first take, so that a
    // slow SM does not set the end.  On smaller batches a block would take
    // about as long as the spread between SMs, and claiming it and refilling
    // the ring cost more than it saves.  The entropy variants have no tail
    // blocks: they run score_rows_kernel, which reads its own range only.
    constexpr int64_t kTailMinShare = 2048, kTailMinBlock = 16;
    p.n_static = p.n_chunks;
    p.tail_chunks = 0;
    p.n_tail = 0;
    const int64_t max_blocks = std::min<int64_t>(8 * warps, scr.max_ranges - 1 - warps);
    if (entropy == nullptr && p.n_chunks >= kTailMinShare * warps && max_blocks > 0) {
        const int64_t tail = p.n_chunks / 16;
        p.tail_chunks = std::max(kTailMinBlock, (tail + max_blocks - 1) / max_blocks);
        p.n_tail = (int32_t)((tail + p.tail_chunks - 1) / p.tail_chunks);
        p.n_static = p.n_chunks - tail;
    }
    const int64_t n_ranges = warps + p.n_tail;
    p.npow = npow;
    p.g = g;
    p.n_taus = n_taus;
    for (int k = 0; k < 4; ++k) p.tau_pow[k] = (tau_pow && k < n_taus) ? tau_pow[k] : 0;
    p.lq_multi = lq_multi;
    p.lp0 = lp0;
    p.lq = lq;
    p.entropy = entropy;
    p.parts = scr.parts;
    p.counters = scr.counters;
    p.claim = scr.counters + n_ranges;
    p.status = status;
    const int n_ctas = (int)((warps + ps::kWarpsPerCta - 1) / ps::kWarpsPerCta);
    // the counters must start at zero whatever the scratch held before
    const size_t zero_bytes = (size_t)((uint8_t *)(p.claim + 1) - (uint8_t *)scr.zero_from);
    ps_status st = map_cuda(cudaMemsetAsync(scr.zero_from, 0, zero_bytes, stream));
    if (st != PS_OK) return st;
    return map_cuda(ps::launch_score_rows(p, n_ctas, stream));
}

// The row kernel on a caller workspace.
ps_status score_rows_launch(const ps_subtree_batch *b, double *lp0, double *lq,
                            double *entropy, int32_t *status, void *workspace,
                            size_t workspace_bytes, void *cuda_stream, int32_t npow, float g,
                            const int32_t *tau_pow, int32_t n_taus, double *lq_multi) {
    const WsLayout wl = ws_layout(b->n_rows, b->n_chains);
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < wl.total)
        return PS_ERR_WORKSPACE;
    if (b->n_rows == 0) return PS_OK;
    int sms = 0;
    ps_status st = device_of(b->logits, &sms);
    if (st != PS_OK) return st;
    uint8_t *ws = (uint8_t *)workspace;
    int32_t *cnt = (int32_t *)(ws + wl.cnt_off);
    const RowsScratch scr{(ps::RowPart *)(ws + wl.parts_off), cnt, ps::kMaxRanges, cnt};
    return launch_rows(b, sms, scr, lp0, lq, entropy, status, cuda_stream, npow, g, tau_pow,
                       n_taus, lq_multi);
}

}  // namespace

extern "C" {

ps_status ps_score_rows(const ps_subtree_batch *b, double *lp0, double *lq, double *entropy,
                        int32_t *status, void *workspace, size_t workspace_bytes,
                        void *cuda_stream) {
    ps_status st = check_batch_host(b);
    if (st != PS_OK) return st;
    if (!lp0 || !lq || !status) return PS_ERR_INVALID_ARG;
    return score_rows_launch(b, lp0, lq, entropy, status, workspace, workspace_bytes,
                             cuda_stream, integer_power(b->tau), (float)(1.0 / b->tau),
                             nullptr, 0, nullptr);
}

ps_status ps_score_rows_multi(const ps_subtree_batch *b, const double *taus, int32_t n_taus,
                              double *lp0, double *lq, double *entropy, int32_t *status,
                              void *workspace, size_t workspace_bytes, void *cuda_stream) {
    ps_status st = check_batch_host(b);
    if (st != PS_OK) return st;
    if (n_taus < 1 || n_taus > 4) return PS_ERR_UNSUPPORTED;
    if (!taus || !lp0 || !lq || !status) return PS_ERR_INVALID_ARG;
    int32_t pw[4], top = 1;
    for (int32_t k = 0; k < n_taus; ++k) {
        if (!(taus[k] > 0.0) || !isfinite(taus[k])) return PS_ERR_INVALID_ARG;
        pw[k] = integer_power(taus[k]);
        if (pw[k] == 0) return PS_ERR_UNSUPPORTED;
        if (pw[k] > top) top = pw[k];
    }
    // the kernel keeps the power sums up to 2^(4y), or up to 2^(8y) when needed
    return score_rows_launch(b, lp0, nullptr, entropy, status, workspace, workspace_bytes,
                             cuda_stream, top == 8 ? 16 : 17, 1.f, pw, n_taus, lq);
}

}  // extern "C"

namespace {

// Host checks of ps_assemble_subtree's arguments.
ps_status check_assemble_host(const ps_subtree_batch *b, const double *lp0, const double *lq,
                              const ps_score_out *out) {
    if (!b || b->T < 1 || b->n_chains < 1 || b->n_seg < b->n_chains || b->n_rows < 0 ||
        !isfinite(b->alpha))
        return PS_ERR_INVALID_ARG;
    if (!b->chain_seg0 || !b->seg_row0 || !b->seg_cut || !b->seg_src) return PS_ERR_INVALID_ARG;
    if (!out || !out->log_accept || !out->status) return PS_ERR_INVALID_ARG;
    if (b->n_rows > 0 && (!lp0 || !lq)) return PS_ERR_INVALID_ARG;
    if ((b->root_lp0 == nullptr) != (b->root_lq == nullptr)) return PS_ERR_INVALID_ARG;
    if (out->eps_class && !(b->eps > 0.0 && b->eps < 0.5)) return PS_ERR_INVALID_ARG;
    return PS_OK;
}

ps::AssembleParams assemble_params(const ps_subtree_batch *b, const double *lp0,
                                   const double *lq, const ps_score_out *out) {
    ps::AssembleParams a{};
    a.T = b->T;
    a.n_chains = b->n_chains;
    a.n_seg = b->n_seg;
    a.n_rows = b->n_rows;
    a.alpha = b->alpha;
    a.chain_seg0 = b->chain_seg0;
    a.seg_row0 = b->seg_row0;
    a.seg_cut = b->seg_cut;
    a.seg_src = b->seg_src;
    a.lp0 = lp0;
    a.lq = lq;
    a.root_lp0 = b->root_lp0;
    a.root_lq = b->root_lq;
    a.lp_y = out->lp_y;
    a.lq_y = out->lq_y;
    a.lp_x = out->lp_x;
    a.lq_x = out->lq_x;
    a.log_ratio = out->log_ratio;
    a.log_accept = out->log_accept;
    a.eps = b->eps;
    a.eps_class = out->eps_class;
    a.status = out->status;
    return a;
}

// Host checks of ps_walk_subtree's arguments.
ps_status check_walk_host(const ps_tree *t, const double *log_accept, const ps_walk_out *out) {
    if (!t || !log_accept || !out) return PS_ERR_INVALID_ARG;
    if (t->n_chains < 1 || t->n_nodes < t->n_chains || t->n_seg < t->n_chains ||
        t->max_steps < 0)
        return PS_ERR_INVALID_ARG;
    if (!t->chain_node0 || !t->chain_seg0 || !t->acc || !t->rej || !t->req || !t->u)
        return PS_ERR_INVALID_ARG;
    if (!out->state_seg || !out->end_node || !out->k_delta || !out->status)
        return PS_ERR_INVALID_ARG;
    return PS_OK;
}

ps::WalkParams walk_params(const ps_tree *t, const double *log_accept, const ps_walk_out *out) {
    ps::WalkParams p{};
    p.n_chains = t->n_chains;
    p.n_nodes = t->n_nodes;
    p.n_seg = t->n_seg;
    p.max_steps = t->max_steps;
    p.chain_node0 = t->chain_node0;
    p.chain_seg0 = t->chain_seg0;
    p.acc = t->acc;
    p.rej = t->rej;
    p.req = t->req;
    p.u = t->u;
    p.log_accept = log_accept;
    p.state_seg = out->state_seg;
    p.end_node = out->end_node;
    p.k_delta = out->k_delta;
    p.path = out->path;
    p.status = out->status;
    return p;
}

}  // namespace

extern "C" {

ps_status ps_assemble_subtree(const ps_subtree_batch *b, const double *lp0, const double *lq,
                              const ps_score_out *out, void *cuda_stream) {
    ps_status st = check_assemble_host(b, lp0, lq, out);
    if (st != PS_OK) return st;
    int sms = 0;
    st = device_of(out->log_accept, &sms);
    if (st != PS_OK) return st;
    return map_cuda(ps::launch_assemble(assemble_params(b, lp0, lq, out),
                                        (cudaStream_t)cuda_stream));
}

ps_status ps_score_subtree(const ps_subtree_batch *b, const ps_score_out *out, void *workspace,
                           size_t workspace_bytes, void *cuda_stream) {
    ps_status st = check_batch_host(b);
    if (st != PS_OK) return st;
    if (!out || !out->log_accept || !out->status) return PS_ERR_INVALID_ARG;
    const WsLayout wl = ws_layout(b->n_rows, b->n_chains);
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < wl.total)
        return PS_ERR_WORKSPACE;
    uint8_t *ws = (uint8_t *)workspace;
    double *lp0 = out->lp0 ? out->lp0 : (double *)(ws + wl.rows_off);
    double *lq = out->lq ? out->lq : (double *)(ws + wl.rows_off) + b->n_rows;
    if (out->eps_class && !(b->eps > 0.0 && b->eps < 0.5)) return PS_ERR_INVALID_ARG;
    st = ps_score_rows(b, lp0, lq, out->entropy, out->status, workspace, workspace_bytes,
                       cuda_stream);
    if (st != PS_OK) return st;
    return ps_assemble_subtree(b, lp0, lq, out, cuda_stream);
}

ps_status ps_walk_subtree(const ps_tree *t, const double *log_accept, const ps_walk_out *out,
                          void *cuda_stream) {
    ps_status st = check_walk_host(t, log_accept, out);
    if (st != PS_OK) return st;
    int sms = 0;
    st = device_of(log_accept, &sms);
    if (st != PS_OK) return st;
    return map_cuda(ps::launch_walk(walk_params(t, log_accept, out), (cudaStream_t)cuda_stream));
}

ps_status ps_score_walk_subtree(const ps_subtree_batch *b, const ps_tree *t,
                                const ps_score_out *out, const ps_walk_out *wout,
                                void *workspace, size_t workspace_bytes, void *cuda_stream) {
    ps_status st = check_batch_host(b);
    if (st != PS_OK) return st;
    if (!out || !out->log_accept || !out->status) return PS_ERR_INVALID_ARG;
    st = check_walk_host(t, out->log_accept, wout);
    if (st != PS_OK) return st;
    if (t->n_chains != b->n_chains || t->n_seg != b->n_seg) return PS_ERR_INVALID_ARG;
    const WsLayout wl = ws_layout(b->n_rows, b->n_chains);
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < wl.total)
        return PS_ERR_WORKSPACE;
    uint8_t *ws = (uint8_t *)workspace;
    double *lp0 = out->lp0 ? out->lp0 : (double *)(ws + wl.rows_off);
    double *lq = out->lq ? out->lq : (double *)(ws + wl.rows_off) + b->n_rows;
    st = check_assemble_host(b, lp0, lq, out);
    if (st != PS_OK) return st;
    int sms = 0;
    st = device_of(b->n_rows > 0 ? b->logits : out->log_accept, &sms);
    if (st != PS_OK) return st;
    cudaStream_t stream = (cudaStream_t)cuda_stream;
    int32_t *chain_cnt = (int32_t *)(ws + wl.chain_cnt_off);
    int32_t *cnt = (int32_t *)(ws + wl.cnt_off);
    if (b->n_rows > 0) {
        // one memset clears the chain counters and the row kernel's counters
        const RowsScratch scr{(ps::RowPart *)(ws + wl.parts_off), cnt, ps::kMaxRanges, chain_cnt};
        st = launch_rows(b, sms, scr, lp0, lq, out->entropy, out->status, cuda_stream,
                         integer_power(b->tau), (float)(1.0 / b->tau), nullptr, 0, nullptr);
    } else {
        st = map_cuda(cudaMemsetAsync(chain_cnt, 0, wl.chain_cnt_bytes, stream));
    }
    if (st != PS_OK) return st;
    // right after the row kernel launched above, the suffix-sum kernel may read
    // the layout before that kernel's results are visible (early)
    return map_cuda(ps::launch_assemble_walk(assemble_params(b, lp0, lq, out),
                                             walk_params(t, out->log_accept, wout), chain_cnt,
                                             b->n_rows > 0, stream));
}

ps_status ps_validate_subtree(const ps_subtree_batch *b, const ps_tree *t, char *msg,
                              size_t msg_len) {
    auto fail = [&](ps_status s, const char *fmt, long long a, long long c) {
        if (msg && msg_len) snprintf(msg, msg_len, fmt, a, c);
        return s;
    };
    if (msg && msg_len) msg[0] = 0;
    if (b) {
        ps_status s = check_batch_host(b, false);
        if (s != PS_OK) return fail(s, "batch header invalid (%lld %lld)", s, 0);
        const int32_t T = b->T;
        if (b->chain_seg0[0] != 0 || b->chain_seg0[b->n_chains] != b->n_seg)
            return fail(PS_ERR_INVALID_ARG, "chain_seg0 must run 0..n_seg (%lld, %lld)",
                        b->chain_seg0[0], b->chain_seg0[b->n_chains]);
        if (b->seg_row0[0] != 0 || b->seg_row0[b->n_seg] != b->n_rows)
            return fail(PS_ERR_INVALID_ARG, "seg_row0 must run 0..n_rows (%lld, %lld)",
                        (long long)b->seg_row0[0], (long long)b->seg_row0[b->n_seg]);
        for (int32_t c = 0; c < b->n_chains; ++c) {
            const int32_t s0 = b->chain_seg0[c], s1 = b->chain_seg0[c + 1];
            if (s1 <= s0) return fail(PS_ERR_INVALID_ARG, "chain %lld has no root (%lld)", c, s1);
            const int32_t rc = b->seg_cut[s0];
            if (b->seg_src[s0] != -1 || rc < 0 || rc > T)
                return fail(PS_ERR_INVALID_ARG, "chain %lld root segment %lld invalid", c, s0);
            for (int32_t s = s0; s < s1; ++s) {
                const int64_t n = b->seg_row0[s + 1] - b->seg_row0[s];
                if (n != (int64_t)(T - b->seg_cut[s]))
                    return fail(PS_ERR_INVALID_ARG, "segment %lld has %lld rows, not T - cut", s, n);
                if (s == s0) continue;
                const int32_t cs = b->seg_cut[s], src = b->seg_src[s];
                if (cs < 0 || cs > T - 1)
                    return fail(PS_ERR_INVALID_ARG, "request %lld cut %lld outside 0..T-1", s, cs);
                if (src < s0 || src >= s1 || src == s)
                    return fail(PS_ERR_INVALID_ARG, "request %lld src %lld not in its chain", s,
                                src);
                const int32_t csrc = src == s0 ? T : b->seg_cut[src];
                if (cs > csrc)
                    return fail(PS_ERR_INFEASIBLE, "request %lld: c_i > c_src (%lld)", s, csrc);
                if (cs < rc && b->root_lp0 == nullptr)
                    return fail(PS_ERR_INFEASIBLE, "request %lld cut below root rows (%lld)", s,
                                rc);
            }
        }
        if (b->tokens && b->n_rows > 0) {
            for (int64_t r = 0; r < b->n_rows; ++r)
                if (b->tokens[r] < 0 || b->tokens[r] >= b->V)
                    return fail(PS_ERR_INVALID_ARG, "row %lld token %lld outside [0, V)", r,
                                b->tokens[r]);
        }
        if (b->row_index && b->n_rows > 0) {
            for (int64_t r = 0; r < b->n_rows; ++r)
                if (b->row_index[r] < 0 || b->row_index[r] >= b->n_logit_rows)
                    return fail(PS_ERR_INVALID_ARG, "row %lld row_index %lld out of range", r,
                                (long long)b->row_index[r]);
        }
    }
    if (t) {
        if (t->n_chains < 1 || t->max_steps < 0 || !t->chain_node0 || !t->chain_seg0 ||
            !t->acc || !t->rej || !t->req)
            return fail(PS_ERR_INVALID_ARG, "tree header invalid (%lld %lld)", t->n_chains,
                        t->max_steps);
        if (b && (t->n_chains != b->n_chains || t->n_seg != b->n_seg))
            return fail(PS_ERR_INVALID_ARG, "tree and batch disagree (%lld chains, %lld segs)",
                        t->n_chains, t->n_seg);
        if (t->chain_node0[0] != 0 || t->chain_node0[t->n_chains] != t->n_nodes)
            return fail(PS_ERR_BAD_TREE, "chain_node0 must run 0..n_nodes (%lld %lld)",
                        t->chain_node0[0], t->chain_node0[t->n_chains]);
        for (int32_t c = 0; c < t->n_chains; ++c) {
            const int32_t n0 = t->chain_node0[c], n1 = t->chain_node0[c + 1];
            const int32_t s0 = t->chain_seg0[c], s1 = t->chain_seg0[c + 1];
            if (n1 <= n0 || s1 <= s0)
                return fail(PS_ERR_BAD_TREE, "chain %lld empty (%lld)", c, n1 - n0);
            // parent count, reachability and state of every node, from the root
            std::vector<int32_t> parents(n1 - n0, 0), state(n1 - n0, -3);
            std::vector<int32_t> used_req(s1 - s0, 0);
            for (int32_t v = n0; v < n1; ++v) {
                const int32_t kids[2] = {t->acc[v], t->rej[v]};
                for (int32_t ch : kids) {
                    if (ch == -1) continue;
                    if (ch <= n0 || ch >= n1)
                        return fail(PS_ERR_BAD_TREE, "node %lld child %lld out of chain", v, ch);
                    if (++parents[ch - n0] > 1)
                        return fail(PS_ERR_BAD_TREE, "node %lld has two parents (%lld)", ch, v);
                }
                const int32_t q = t->req[v];
                if (q >= 0) {
                    if (q <= s0 || q >= s1)
                        return fail(PS_ERR_BAD_TREE, "node %lld request %lld not in chain", v, q);
                    if (used_req[q - s0]++)
                        return fail(PS_ERR_BAD_TREE, "request %lld used twice (node %lld)", q, v);
                    if (t->acc[v] < 0 || t->rej[v] < 0)
                        return fail(PS_ERR_BAD_TREE, "node %lld has a request but no children %lld",
                                    v, q);
                } else if (q != PS_NODE_LEAF && q != PS_NODE_DEFERRED) {
                    return fail(PS_ERR_BAD_TREE, "node %lld request code %lld invalid", v, q);
                }
            }
            if (parents[0] != 0) return fail(PS_ERR_BAD_TREE, "root of chain %lld has a parent %lld", c, 0);
            // forward pass in an order where parents come first
            std::vector<int32_t> order;
            order.push_back(n0);
            state[0] = s0;
            for (size_t i = 0; i < order.size(); ++i) {
                const int32_t v = order[i];
                const int32_t q = t->req[v];
                if (t->rej[v] >= 0) {
                    state[t->rej[v] - n0] = state[v - n0];
                    order.push_back(t->rej[v]);
                }
                if (t->acc[v] >= 0) {
                    state[t->acc[v] - n0] = q >= 0 ? q : -2;   // -2: no generated state
                    if (q >= 0) order.push_back(t->acc[v]);
                    if (b && q >= 0 && b->seg_src[q] != state[v - n0])
                        return fail(PS_ERR_BAD_TREE,
                                    "request %lld: seg_src is not its decision node's state %lld",
                                    q, state[v - n0]);
                }
            }
            for (int32_t v = n0; v < n1; ++v)
                if (state[v - n0] == -3)
                    return fail(PS_ERR_BAD_TREE, "node %lld unreachable from the root (%lld)", v, c);
        }
    }
    return PS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Scoring without a caller workspace: scratch lives in one static device array
// ---------------------------------------------------------------------------
namespace {
constexpr int64_t kNoAllocMaxRows = 262144;     // per-row values kept in the array
constexpr int kNoAllocMaxRanges = 4096;          // chunk ranges: split-row partials, counters
constexpr size_t kNoAllocRowBytes = (size_t)kNoAllocMaxRows * 2 * sizeof(double);
constexpr size_t kNoAllocPartBytes = (size_t)2 * kNoAllocMaxRanges * sizeof(ps::RowPart);
constexpr size_t kNoAllocCntBytes = (size_t)kNoAllocMaxRanges * sizeof(int32_t);
constexpr size_t kNoAllocBytes = kNoAllocRowBytes + kNoAllocPartBytes + kNoAllocCntBytes;
}  // namespace

// About 4.5 MB on every device that loads the library.  Host code must not use
// this name as an address: it is a host-side stand-in; the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char ps_noalloc_scratch[kNoAllocBytes];

namespace {
// Device address of ps_noalloc_scratch on device `dev` (which the caller has
// made current); looked up once per device.
ps_status noalloc_scratch(int dev, uint8_t **out) {
    static std::mutex mu;
    static std::vector<void *> addr;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)addr.size() <= dev) addr.resize(dev + 1, nullptr);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, ps_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return PS_ERR_CUDA;
        }
        addr[dev] = p;
    }
    *out = (uint8_t *)addr[dev];
    return PS_OK;
}
}  // namespace

extern "C" ps_status ps_score_subtree_noalloc(const ps_subtree_batch *b, const ps_score_out *out,
                                              void *cuda_stream) {
    ps_status st = check_batch_host(b);
    if (st != PS_OK) return st;
    if (!out || !out->log_accept || !out->status) return PS_ERR_INVALID_ARG;
    if (out->eps_class && !(b->eps > 0.0 && b->eps < 0.5)) return PS_ERR_INVALID_ARG;
    // a per-row array the caller does not supply is kept in the static array
    const bool lp0_scratch = out->lp0 == nullptr, lq_scratch = out->lq == nullptr;
    if ((lp0_scratch || lq_scratch) && b->n_rows > kNoAllocMaxRows) return PS_ERR_WORKSPACE;
    int sms = 0;
    st = device_of(b->n_rows > 0 ? b->logits : out->log_accept, &sms);
    if (st != PS_OK) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return PS_ERR_CUDA;
    uint8_t *base = nullptr;
    st = noalloc_scratch(dev, &base);
    if (st != PS_OK) return st;
    double *lp0 = lp0_scratch ? (double *)base : out->lp0;
    double *lq = lq_scratch ? (double *)base + kNoAllocMaxRows : out->lq;
    if (b->n_rows > 0) {
        int32_t *cnt = (int32_t *)(base + kNoAllocRowBytes + kNoAllocPartBytes);
        const RowsScratch scr{(ps::RowPart *)(base + kNoAllocRowBytes), cnt, kNoAllocMaxRanges,
                              cnt};
        st = launch_rows(b, sms, scr, lp0, lq, out->entropy, out->status, cuda_stream,
                         integer_power(b->tau), (float)(1.0 / b->tau), nullptr, 0, nullptr);
        if (st != PS_OK) return st;
    }
    return ps_assemble_subtree(b, lp0, lq, out, cuda_stream);
}

extern "C" ps_status ps_selftest_wait_timeout(uint64_t limit_ns, int32_t *status, void *cuda_stream) {
    if (limit_ns < 1000ull || limit_ns > 2000000000ull) return PS_ERR_INVALID_ARG;
    if (!status) return PS_ERR_INVALID_ARG;
    int sms = 0;
    ps_status st = device_of(status, &sms);
    if (st != PS_OK) return st;
    return map_cuda(ps::launch_wait_selftest(limit_ns, status, (cudaStream_t)cuda_stream));
}

extern "C" ps_status ps_selftest_read(const void *data, size_t bytes, uint32_t *sink,
                                      void *cuda_stream) {
    if (!data || !sink || !aligned(data, 16) || bytes % 16 != 0) return PS_ERR_INVALID_ARG;
    int sms = 0;
    ps_status st = device_of(data, &sms);
    if (st != PS_OK) return st;
    return map_cuda(ps::launch_read_probe(data, (int64_t)(bytes / 16), sink, sms,
                                          (cudaStream_t)cuda_stream));
}

extern "C" ps_status ps_carry_state(const ps_subtree_batch *b, const ps_carry_io *io,
                                      void *cuda_stream) {
    if (!b || !io || b->T < 1 || b->n_chains < 1 || b->n_seg < b->n_chains || b->n_rows < 0)
        return PS_ERR_INVALID_ARG;
    if (!b->chain_seg0 || !b->seg_row0 || !b->seg_cut || !b->seg_src) return PS_ERR_INVALID_ARG;
    if (!io->state_seg || !io->next_lp0 || !io->next_lq || !io->status) return PS_ERR_INVALID_ARG;
    if (b->n_rows > 0 && (!io->row_lp0 || !io->row_lq)) return PS_ERR_INVALID_ARG;
    if (io->next_entropy && b->n_rows > 0 && !io->row_entropy) return PS_ERR_INVALID_ARG;
    if (io->confidence && !io->next_entropy) return PS_ERR_INVALID_ARG;
    int sms = 0;
    ps_status st = device_of(io->next_lp0, &sms);
    if (st != PS_OK) return st;
    ps::CarryParams p;
    p.T = b->T;
    p.n_chains = b->n_chains;
    p.n_seg = b->n_seg;
    p.n_rows = b->n_rows;
    p.chain_seg0 = b->chain_seg0;
    p.seg_row0 = b->seg_row0;
    p.seg_cut = b->seg_cut;
    p.seg_src = b->seg_src;
    p.io = *io;
    return map_cuda(ps::launch_carry(p, (cudaStream_t)cuda_stream));
}
