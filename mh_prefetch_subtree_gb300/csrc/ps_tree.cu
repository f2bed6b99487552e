// Host-side construction of prefetched subtrees (PreSTO section 3.2 step (1)
// and Appendix C): BFS request collection under Condition 1, and the
// predictive allocation of Appendix C.3-C.4.  No device code.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "ps_internal.cuh"

extern "C" double ps_midpoint_branch_probability(double p_accept, double p_reject) {
    // eq. (14): the midpoint of the interval Lemma 3 puts around E[h(v+)]
    return 0.5 * (1.0 + p_accept - p_reject);
}

extern "C" ps_status ps_build_bfs_tree(int32_t T, int32_t n_pf, int32_t depth_cap,
                                       const int32_t *cuts, int32_t n_cuts, int32_t max_nodes,
                                       int32_t max_seg, int32_t *acc, int32_t *rej, int32_t *req,
                                       int32_t *node_cut, int32_t *deferred_cut,
                                       int32_t *seg_cut, int32_t *seg_src, int32_t *n_nodes_out,
                                       int32_t *n_seg_out, int32_t *n_cuts_used) {
    if (T < 1 || n_pf < 0 || n_cuts < 0 || max_nodes < 1 || max_seg < 1) return PS_ERR_INVALID_ARG;
    if (!acc || !rej || !req || !node_cut || !deferred_cut || !seg_cut || !seg_src ||
        !n_nodes_out || !n_seg_out || !n_cuts_used || (n_cuts > 0 && !cuts))
        return PS_ERR_INVALID_ARG;
    std::vector<int32_t> depth(1, 0), state(1, 0), queue(1, 0);
    int32_t nn = 1, ns = 1, used = 0;
    acc[0] = rej[0] = req[0] = -1;
    node_cut[0] = T;
    deferred_cut[0] = -1;
    seg_cut[0] = T;
    seg_src[0] = -1;
    size_t head = 0;
    while (head < queue.size() && ns - 1 < n_pf) {
        const int32_t v = queue[head++];
        if (depth_cap >= 0 && depth[v] >= depth_cap) continue;
        if (used >= n_cuts) break;                   // no more drawn cuts: stop here
        const int32_t c = cuts[used++];
        if (c < 0 || c > T - 1) return PS_ERR_INVALID_ARG;
        if (nn + 2 > max_nodes) return PS_ERR_INVALID_ARG;
        const int32_t a = nn, b = nn + 1;
        nn += 2;
        for (int32_t x : {a, b}) {
            acc[x] = rej[x] = req[x] = -1;
            deferred_cut[x] = -1;
            depth.push_back(depth[v] + 1);
        }
        node_cut[a] = c;
        node_cut[b] = node_cut[v];                   // a rejection keeps the cut
        acc[v] = a;
        rej[v] = b;
        state.push_back(-1);
        state.push_back(state[v]);                   // and the state
        if (c <= node_cut[v]) {                      // Condition 1: feasible now
            if (ns + 1 > max_seg) return PS_ERR_INVALID_ARG;
            seg_cut[ns] = c;
            seg_src[ns] = state[v];
            req[v] = ns;
            state[a] = ns;
            ++ns;
            queue.push_back(a);
        } else {                                     // deferred, keeps its cut
            req[v] = PS_NODE_DEFERRED;
            deferred_cut[v] = c;
        }
        queue.push_back(b);                          // enqueued either way
    }
    int32_t rc = T;
    for (int32_t s = 1; s < ns; ++s) rc = std::min(rc, seg_cut[s]);
    seg_cut[0] = rc;                                 // root rows the requests need
    *n_nodes_out = nn;
    *n_seg_out = ns;
    *n_cuts_used = used;
    return PS_OK;
}

extern "C" ps_status ps_predictive_allocation(int32_t n_nodes, const int32_t *acc,
                                              const int32_t *rej, const uint8_t *candidate,
                                              const double *h_acc, int32_t budget,
                                              double *value, uint8_t *selected) {
    if (n_nodes < 1 || budget < 0 || !acc || !rej || !candidate || !h_acc || !value || !selected)
        return PS_ERR_INVALID_ARG;
    for (int32_t v = 0; v < n_nodes; ++v)
        if (!(h_acc[v] >= 0.0 && h_acc[v] <= 1.0)) return PS_ERR_INVALID_ARG;
    // the tree: children in range, one parent each, the root has none
    std::vector<uint8_t> has_parent(n_nodes, 0);
    for (int32_t v = 0; v < n_nodes; ++v)
        for (int32_t ch : {acc[v], rej[v]}) {
            if (ch == -1) continue;
            if (ch <= 0 || ch >= n_nodes || has_parent[ch]) return PS_ERR_BAD_TREE;
            has_parent[ch] = 1;
        }
    // post-order from the root (children before parents)
    std::vector<int32_t> order;
    order.reserve(n_nodes);
    std::vector<int32_t> stack(1, 0);
    while (!stack.empty()) {
        const int32_t v = stack.back();
        stack.pop_back();
        order.push_back(v);
        for (int32_t ch : {acc[v], rej[v]})
            if (ch >= 0) stack.push_back(ch);
    }
    const size_t B = (size_t)budget + 1;
    std::vector<double> V;
    std::vector<int32_t> arg;
    try {
        V.assign((size_t)n_nodes * B, 0.0);
        arg.assign((size_t)n_nodes * B, -1);
    } catch (const std::bad_alloc &) {
        return PS_ERR_UNSUPPORTED;
    }
    auto val = [&](int32_t v, int32_t b) -> double { return v < 0 ? 0.0 : V[(size_t)v * B + b]; };
    for (size_t i = order.size(); i-- > 0;) {
        const int32_t v = order[i];
        if (!candidate[v]) continue;                  // V(v, b) = 0
        const double h = h_acc[v];
        for (int32_t b = 1; b <= budget; ++b) {
            // eq. (19): one request expands v, the other b-1 are split m / b-1-m
            double best = -1.0;
            int32_t am = -1;
            for (int32_t m = 0; m < b; ++m) {
                const double x = h * val(acc[v], m) + (1.0 - h) * val(rej[v], b - 1 - m);
                if (x > best) {
                    best = x;
                    am = m;
                }
            }
            V[(size_t)v * B + b] = 1.0 + best;
            arg[(size_t)v * B + b] = am;
        }
    }
    memset(selected, 0, (size_t)n_nodes);
    std::vector<std::pair<int32_t, int32_t>> st(1, {0, budget});
    while (!st.empty()) {
        const auto [v, b] = st.back();
        st.pop_back();
        if (v < 0 || b == 0 || !candidate[v]) continue;
        selected[v] = 1;
        const int32_t m = arg[(size_t)v * B + b];
        st.push_back({acc[v], m});
        st.push_back({rej[v], b - 1 - m});
    }
    *value = val(0, budget);
    return PS_OK;
}
