"""libps's host-side tree construction against the oracle (CPU only):
BFS request collection (section 3.2 step (1)) and the predictive allocation
dynamic program (eq. (19))."""

import numpy as np
import pytest

import mh_prefetch_subtree_gb300 as ps
from oracle import trees as OT
from tests.test_oracle_trees import _random_candidate_tree


@pytest.fixture(scope="module", autouse=True)
def built():
    from mh_prefetch_subtree_gb300.build import build
    build()


def test_bfs_matches_oracle():
    rng = np.random.default_rng(5)
    for _ in range(300):
        T = int(rng.integers(1, 80))
        n_pf = int(rng.integers(0, 20))
        cap = None if rng.random() < 0.5 else int(rng.integers(1, 6))
        cuts = rng.integers(0, T, int(rng.integers(0, 120))).astype(np.int32)
        g = ps.ps_build_bfs_tree(T, n_pf, cap, cuts)
        o = OT.bfs(T, n_pf, cap, cuts)
        for k in ("acc", "rej", "req", "node_cut", "seg_cut", "seg_src"):
            assert np.array_equal(g[k], o[k]), k
        assert g["cuts_used"] == o["cuts_used"]
        d = {v: c for v, c in enumerate(g["deferred_cut"]) if c >= 0}
        assert d == o["deferred"]


def test_bfs_tree_validates_and_rejects_bad_cuts():
    g = ps.ps_build_bfs_tree(10, 3, None, [4, 2, 9, 1])
    assert g["seg_cut"][0] == min(g["seg_cut"][1:])
    with pytest.raises(ps.PsError):
        ps.ps_build_bfs_tree(10, 3, None, [4, 10])


def test_allocation_matches_oracle_dp():
    rng = np.random.default_rng(6)
    for _ in range(80):
        acc, rej, cand, h = _random_candidate_tree(rng, int(rng.integers(1, 7)))
        for budget in (0, 1, 3, 8, 20):
            v, sel = ps.ps_predictive_allocation(acc, rej, cand, h, budget)
            vo, selo = OT.allocation_dp(acc, rej, cand, h, budget)
            assert abs(v - vo) <= 1e-12 * max(1.0, vo)
            assert np.array_equal(sel, selo)


def test_allocation_is_best_first_by_reaching_weight():
    # with 0 < h < 1 the reaching weight strictly falls along every path, so
    # the optimum of eq. (17) is the budget's best candidates by R (Lemma 1)
    rng = np.random.default_rng(7)
    for _ in range(40):
        acc, rej, cand, h = _random_candidate_tree(rng, 6)
        R = OT.reaching_weights(acc, rej, h)
        # candidates whose whole path is candidate
        ok = np.zeros(len(acc), bool)
        order = [0]
        ok[0] = cand[0]
        for v in order:
            for ch in (acc[v], rej[v]):
                if ch >= 0:
                    ok[ch] = ok[v] and cand[ch]
                    order.append(ch)
        for budget in (1, 4, 10):
            v, sel = ps.ps_predictive_allocation(acc, rej, cand, h, budget)
            top = np.sort(R[ok])[::-1][:budget]
            assert abs(v - top.sum()) <= 1e-12


def test_midpoint():
    assert ps.ps_midpoint_branch_probability(0.6, 0.1) == OT.midpoint_h(0.6, 0.1)


def test_allocation_rejects_bad_trees():
    with pytest.raises(ps.PsError):
        ps.ps_predictive_allocation([1, -1], [1, -1], [1, 1], [0.5, 0.5], 2)   # two parents
    with pytest.raises(ps.PsError):
        ps.ps_predictive_allocation([-1], [-1], [1], [1.5], 2)                  # h outside [0,1]
