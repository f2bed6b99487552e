"""Pins for the oracle's tree construction: BFS against the pages' Example 2
and Condition 1, the allocation DP against brute force (Proposition 2), the
Lemma 1 identity, and the midpoint rule (eq. (14))."""

import json
import os

import numpy as np

from oracle import trees as OT

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_bfs_example2():
    with open(os.path.join(GOLDEN, "example2_bfs.json")) as fh:
        g = json.load(fh)
    T, c1, c2 = 20, 11, 6
    t = OT.bfs(T, g["n_pf"], None, [c1, c2])
    assert t["acc"][0] == 1 and t["acc"][1] == 3 and t["rej"][0] == 2
    assert list(t["seg_cut"][1:]) == [c1, c2] and list(t["seg_src"][1:]) == [0, 1]
    assert t["req"][0] == 1 and t["req"][1] == 2 and t["node_cut"][0] == T


def test_bfs_condition1_and_deferral():
    rng = np.random.default_rng(1)
    for _ in range(300):
        T = int(rng.integers(1, 50))
        cuts = rng.integers(0, T, 200)
        t = OT.bfs(T, int(rng.integers(0, 15)), None if rng.random() < .5 else 4, cuts)
        for v, r in enumerate(t["req"]):
            if r >= 0:
                assert t["seg_cut"][r] <= t["node_cut"][v]                 # Condition 1
                src = t["seg_src"][r]
                c_src = T if src == 0 else t["seg_cut"][src]
                assert t["seg_cut"][r] <= c_src
            elif r == -2:
                assert t["deferred"][v] > t["node_cut"][v]
        # a rejection child keeps its parent's cut
        for v in range(len(t["acc"])):
            if t["rej"][v] >= 0:
                assert t["node_cut"][t["rej"][v]] == t["node_cut"][v]


def _random_candidate_tree(rng, depth):
    acc, rej = [-1], [-1]
    frontier = [(0, 0)]
    while frontier:
        v, d = frontier.pop()
        if d < depth and rng.random() < 0.85:
            a, b = len(acc), len(acc) + 1
            acc += [-1, -1]
            rej += [-1, -1]
            acc[v], rej[v] = a, b
            frontier += [(a, d + 1), (b, d + 1)]
    n = len(acc)
    cand = rng.random(n) < 0.8
    cand[0] = True
    h = rng.uniform(0.02, 0.98, n)
    return np.array(acc), np.array(rej), cand, h


def test_dp_equals_brute_force():
    rng = np.random.default_rng(2)
    for _ in range(60):
        acc, rej, cand, h = _random_candidate_tree(rng, 3)
        for budget in range(0, 6):
            v, sel = OT.allocation_dp(acc, rej, cand, h, budget)
            b = OT.allocation_brute(acc, rej, cand, h, budget)
            assert abs(v - b) <= 1e-12
            # the selection is ancestor-closed, within budget, and attains V (Lemma 1)
            R = OT.reaching_weights(acc, rej, h)
            assert sel.sum() <= budget and np.all(cand[sel])
            assert abs(R[sel].sum() - v) <= 1e-12


def test_dp_on_a_chain_closed_form():
    # a unary chain of rejections, h = 0.3 everywhere: V(v0, b) = sum_{k<b} 0.7^k
    n = 12
    acc = np.full(n, -1)
    rej = np.array([i + 1 if i + 1 < n else -1 for i in range(n)])
    h = np.full(n, 0.3)
    cand = np.ones(n, dtype=bool)
    for b in range(0, n + 3):
        v, _ = OT.allocation_dp(acc, rej, cand, h, b)
        assert abs(v - sum(0.7 ** k for k in range(min(b, n)))) <= 1e-12


def test_midpoint_rule():
    assert OT.midpoint_h(1.0, 0.0) == 1.0
    assert OT.midpoint_h(0.0, 1.0) == 0.0
    assert OT.midpoint_h(0.0, 0.0) == 0.5
    assert abs(OT.midpoint_h(0.6, 0.1) - (0.6 + 0.5 * 0.3)) <= 1e-15
