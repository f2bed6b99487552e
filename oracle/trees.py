"""CPU oracle for building prefetching trees.  TEST INFRASTRUCTURE: only the
tests may import it; it shares no code with libps or with the input
generator.

From "PreSTO: Predictive Subtree Prefetching for Fast LLM Power Sampling":

* ``bfs``                 BFS request collection with deferral (section 3.2
                          step (1), Example 2, Condition 1, the K - k depth cap
                          of Appendix C.1); the cut of each expansion is an
                          input (Proposition 1, (A2));
* ``midpoint_h``          predicted branch probability from class
                          probabilities (eq. (14), Lemma 3);
* ``allocation_dp``       the dynamic program of eq. (19) (Proposition 2),
                          written as a memoised recursion;
* ``allocation_brute``    the maximum of eq. (17) by enumerating every
                          ancestor-closed selection (small trees);
* ``reaching_weights``    R(v) of eq. (11).
"""

from __future__ import annotations

import itertools
from collections import deque
from functools import lru_cache

import numpy as np


def bfs(T: int, n_pf: int, depth_cap: int | None, cuts) -> dict:
    """Nodes are numbered in creation order, root 0.  Each expansion of a node
    v draws the next cut c from `cuts`; the acceptance child gets cut c, the
    rejection child v's cut; the request is feasible when c <= cut(v).  A
    feasible request's acceptance child is enqueued; the rejection child is
    always enqueued.  The root's cut is T."""
    cuts = list(cuts)
    acc, rej, req, node_cut, depth = [-1], [-1], [-1], [T], [0]
    state = [0]                        # segment of each node's state (0 = root)
    seg_cut, seg_src = [T], [-1]
    deferred = {}
    used = 0
    q = deque([0])
    while q and len(seg_cut) - 1 < n_pf:
        v = q.popleft()
        if depth_cap is not None and depth[v] >= depth_cap:
            continue
        if used >= len(cuts):          # no more drawn cuts: stop
            break
        c = int(cuts[used])
        used += 1
        a, b = len(acc), len(acc) + 1
        for _ in range(2):
            acc.append(-1)
            rej.append(-1)
            req.append(-1)
            depth.append(depth[v] + 1)
        node_cut += [c, node_cut[v]]
        acc[v], rej[v] = a, b
        if c <= node_cut[v]:
            seg_cut.append(c)
            seg_src.append(state[v])
            req[v] = len(seg_cut) - 1
            state += [req[v], state[v]]
            q.append(a)
        else:
            req[v] = -2
            deferred[v] = c
            state += [-1, state[v]]
        q.append(b)
    if len(seg_cut) > 1:
        seg_cut[0] = min(seg_cut[1:])
    return dict(acc=np.array(acc, np.int32), rej=np.array(rej, np.int32),
                req=np.array(req, np.int32), node_cut=np.array(node_cut, np.int32),
                seg_cut=np.array(seg_cut, np.int32), seg_src=np.array(seg_src, np.int32),
                deferred=deferred, cuts_used=used)


def midpoint_h(p_accept: float, p_reject: float) -> float:
    """eq. (14): h(v+) = 1/2 [1 + P(certain accept) - P(certain reject)]."""
    return 0.5 * (1.0 + p_accept - p_reject)


def reaching_weights(acc, rej, h):
    """eq. (11): R(v0) = 1, R(v+) = R(v) h(v+), R(v-) = R(v) (1 - h(v+))."""
    R = np.zeros(len(acc))
    R[0] = 1.0
    order = [0]
    for v in order:
        for ch, w in ((acc[v], h[v]), (rej[v], 1.0 - h[v])):
            if ch >= 0:
                R[ch] = R[v] * w
                order.append(int(ch))
    return R


def allocation_dp(acc, rej, candidate, h, budget: int):
    """eq. (19): V(v, b) = 0 if v is not a candidate or b = 0, else
    1 + max_{0 <= m <= b-1} { h V(v+, m) + (1 - h) V(v-, b-1-m) }.
    Returns V(v0, budget) and the selection that attains it (smallest m on ties)."""
    acc = [int(x) for x in acc]
    rej = [int(x) for x in rej]

    @lru_cache(maxsize=None)
    def V(v: int, b: int):
        if v < 0 or b == 0 or not candidate[v]:
            return 0.0, -1
        best, arg = -1.0, -1
        for m in range(b):
            val = h[v] * V(acc[v], m)[0] + (1.0 - h[v]) * V(rej[v], b - 1 - m)[0]
            if val > best:
                best, arg = val, m
        return 1.0 + best, arg

    sel = np.zeros(len(acc), dtype=bool)
    stack = [(0, budget)]
    while stack:
        v, b = stack.pop()
        if v < 0 or b == 0 or not candidate[v]:
            continue
        sel[v] = True
        m = V(v, b)[1]
        stack.append((acc[v], m))
        stack.append((rej[v], b - 1 - m))
    return V(0, budget)[0], sel


def allocation_brute(acc, rej, candidate, h, budget: int):
    """max over ancestor-closed selections I of candidate nodes, |I| <= budget,
    of sum_{v in I} R(v) (eq. (17) with Lemma 1)."""
    n = len(acc)
    R = reaching_weights(acc, rej, h)
    parent = np.full(n, -1)
    for v in range(n):
        for ch in (acc[v], rej[v]):
            if ch >= 0:
                parent[ch] = v
    cand = [v for v in range(n) if candidate[v]]
    best = 0.0
    for k in range(0, min(budget, len(cand)) + 1):
        for sub in itertools.combinations(cand, k):
            s = set(sub)
            if all(v == 0 or parent[v] in s for v in s):
                best = max(best, float(sum(R[v] for v in s)))
    return best
