// The MH walk of one chain by one warp (PreSTO section 3.2 step (3); Example 5;
// Algorithm 2, MHTransition), shared by the walk kernel and the fused
// suffix-sum + walk kernel.
//
// The warp copies the chain's node arrays and its requests' uniforms into
// shared memory with coalesced loads (when the chain fits), the lanes take
// every request's accept/reject decision at once, then lane 0 walks: at a
// node whose request was scored it completes one transition, moving to the
// acceptance child when u <= A = exp(log A) and to the rejection child
// otherwise; it stops at a leaf, at a node whose request was deferred, or
// after max_steps transitions.  The walk is bounded by the chain's node count
// as well, so a cyclic tree cannot loop; every id is range-checked and a bad
// one ends the walk with a status bit.
#pragma once

#include <math.h>

#include "ps_internal.cuh"

namespace ps {
namespace {

constexpr int kNodeCap = 512;   // nodes per chain held in shared memory
constexpr int kSegCap = 256;    // segments per chain held in shared memory

struct WalkSmem {
    int32_t acc[kNodeCap];
    int32_t rej[kNodeCap];
    int32_t req[kNodeCap];
    int8_t acc_dec[kSegCap];    // decide(u, log A) of each request of the chain
    double u[kSegCap];
};

// The accept test of Algorithm 1, u <= A with A = exp(log A): 1 accept,
// 0 reject, -1 the uniform is outside (0, 1].  A float exponential settles it
// unless u is within 1e-5 (relative) of A; below log A = -80, A < 1.9e-35, so
// every u >= 1e-30 rejects.  Only the rest (a near tie, or a tiny u) takes the
// float64 exponential, which is slow on this GPU's float64 pipe.  A NaN log A
// rejects.
__device__ __forceinline__ int8_t decide(double u, double la) {
    if (!(u > 0.0 && u <= 1.0)) return -1;
    if (!(la == la)) return 0;
    if (la >= 0.0) return 1;
    if (la > -80.0) {
        // expf is within 2 ulps; rounding la to float moves the exponent by at
        // most 80 * 2^-24, so a is within 5e-6 of A (relative)
        const double a = (double)expf((float)la);
        if (u < a * (1.0 - 1e-5)) return 1;
        if (u > a * (1.0 + 1e-5)) return 0;
    } else if (u >= 1e-30) {
        return 0;
    }
    return u <= exp(la) ? 1 : 0;
}

// Chain c's bounds and, when the chain fits, its node arrays and its
// requests' uniforms in shared memory.  All 32 lanes call it and get the same
// result; the copies are visible to the warp after a __syncwarp().
struct ChainStage {
    int32_t n0, n1, s0, s1;
    bool ok;        // the bounds are consistent
    bool staged;    // the node arrays and uniforms are in shared memory
};

__device__ __forceinline__ ChainStage stage_chain(const WalkParams &p, int c, WalkSmem &w,
                                                  int lane) {
    ChainStage g;
    g.n0 = p.chain_node0[c];
    g.n1 = p.chain_node0[c + 1];
    g.s0 = p.chain_seg0[c];
    g.s1 = p.chain_seg0[c + 1];
    g.ok = !(g.n0 < 0 || g.n1 > p.n_nodes || g.n1 <= g.n0 || g.s0 < 0 || g.s1 > p.n_seg ||
             g.s1 <= g.s0);
    g.staged = g.ok && g.n1 - g.n0 <= kNodeCap && g.s1 - g.s0 <= kSegCap;
    if (g.staged) {
        for (int i = lane; i < g.n1 - g.n0; i += 32) {
            w.acc[i] = p.acc[g.n0 + i];
            w.rej[i] = p.rej[g.n0 + i];
            w.req[i] = p.req[g.n0 + i];
        }
        for (int i = lane; i < g.s1 - g.s0; i += 32) w.u[i] = p.u[g.s0 + i];
    }
    return g;
}

// Walks chain c (0 <= c < n_chains) with the calling warp, given what
// stage_chain() returned for it; all 32 lanes call it, after log A is visible
// to them.
__device__ __forceinline__ void walk_staged(const WalkParams &p, int c, const ChainStage &g,
                                            WalkSmem &w, int lane) {
    const int stride = p.max_steps + 1;
    int32_t *path = p.path ? p.path + (int64_t)c * stride : nullptr;
    const int32_t n0 = g.n0, n1 = g.n1, s0 = g.s0, s1 = g.s1;
    if (!g.ok) {
        if (lane == 0) {
            set_status(p.status, PS_DEV_BAD_TREE);
            p.state_seg[c] = -1;
            p.end_node[c] = -1;
            p.k_delta[c] = 0;
        }
        if (path)
            for (int i = lane; i < stride; i += 32) path[i] = -1;
        return;
    }
    const int32_t nn = n1 - n0;
    const bool staged = g.staged;
    if (staged) {
        // each request's decision, taken by all lanes at once so that the walk
        // below only follows it (a lane reads the uniforms it staged itself)
        for (int i = lane; i < s1 - s0; i += 32)
            w.acc_dec[i] = decide(w.u[i], __ldcg(p.log_accept + s0 + i));
    }
    if (path)
        for (int i = lane; i < stride; i += 32) path[i] = -1;
    __syncwarp();
    if (lane != 0) return;

    auto ACC = [&](int32_t v) { return staged ? w.acc[v - n0] : p.acc[v]; };
    auto REJ = [&](int32_t v) { return staged ? w.rej[v - n0] : p.rej[v]; };
    auto REQ = [&](int32_t v) { return staged ? w.req[v - n0] : p.req[v]; };
    auto DECISION = [&](int32_t s) {
        return staged ? w.acc_dec[s - s0] : decide(p.u[s], __ldcg(p.log_accept + s));
    };

    int32_t v = n0;
    int32_t state = s0;
    int32_t k = 0;
    int32_t bits = 0;
    if (path) path[0] = v;
    const int32_t bound = min(p.max_steps, nn);
    while (k < bound) {
        const int32_t s = REQ(v);
        if (s == PS_NODE_LEAF || s == PS_NODE_DEFERRED) break;
        if (s <= s0 || s >= s1) {          // not a request of this chain
            bits |= PS_DEV_BAD_TREE;
            break;
        }
        const int8_t dec = DECISION(s);
        const bool accept = dec == 1;
        if (dec < 0) bits |= PS_DEV_BAD_UNIFORM;
        const int32_t nv = accept ? ACC(v) : REJ(v);
        if (nv < n0 || nv >= n1) {
            bits |= PS_DEV_BAD_TREE;
            break;
        }
        ++k;
        if (accept) state = s;
        v = nv;
        if (path) path[k] = v;
    }
    // more transitions than nodes can only come from a cycle
    if (k == nn && k < p.max_steps && REQ(v) >= 0) bits |= PS_DEV_BAD_TREE;
    if (bits) set_status(p.status, bits);
    p.state_seg[c] = state;
    p.end_node[c] = v;
    p.k_delta[c] = k;
}

// Stages and walks chain c in one go (all 32 lanes call it).
__device__ __forceinline__ void walk_chain(const WalkParams &p, int c, WalkSmem &w, int lane) {
    const ChainStage g = stage_chain(p, c, w, lane);
    walk_staged(p, c, g, w, lane);
}

}  // namespace
}  // namespace ps
