"""Planted mistakes in the oracle's entropy, epsilon classes, carry-over and
tree construction (on the CPU): each pin must catch its own, and the
unmodified oracle passes every pin."""

import numpy as np
import pytest

import oracle
from oracle import trees as OT
from tests import pins


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def _oracle_entropy(x):
    V = x.shape[1]
    tok = np.zeros(x.shape[0], np.int32)
    return oracle.row_logprobs(np.ascontiguousarray(x, np.float32), "f32", V, tok, 1.0,
                               entropy=True)[2]


def _entropy_parts(x):
    """m, j*, E = sum_{j != j*} e^(l_j - m) and sum_{j != j*} e^(l_j - m)(l_j - m)."""
    x = x.astype(np.float64)
    m = x.max(axis=1, keepdims=True)
    d = x - m
    e = np.exp(d)
    js = x.argmax(axis=1)
    i = np.arange(x.shape[0])
    e[i, js] = 0.0
    ed = e * np.where(e > 0, d, 0.0)              # -inf entries have e = 0
    return e.sum(1), ed.sum(1)


def test_unmodified_oracle_passes_the_next_row_pins():
    pins.pin_entropy_library(_oracle_entropy)
    pins.pin_entropy_uniform(_oracle_entropy)
    pins.pin_eps_classes(oracle.eps_class)
    pins.pin_carry_example5(oracle.carry_state)
    pins.pin_bfs_example2(OT.bfs)
    pins.pin_bfs_condition1(OT.bfs, trials=100)
    pins.pin_dp_brute_force(OT.allocation_dp, OT.allocation_brute, OT.reaching_weights,
                            trials=20)


def test_entropy_without_the_normaliser_is_caught():
    def bad(x):
        E, A = _entropy_parts(x)
        return np.log1p(E) - A                      # the / (1 + E) dropped
    _fails(pins.pin_entropy_library, bad)


def test_entropy_sign_error_is_caught():
    def bad(x):
        E, A = _entropy_parts(x)
        return np.log1p(E) + A / (1.0 + E)
    _fails(pins.pin_entropy_library, bad)


def test_entropy_in_bits_is_caught():
    def bad(x):
        E, A = _entropy_parts(x)
        return (np.log1p(E) - A / (1.0 + E)) / np.log(2.0)
    _fails(pins.pin_entropy_uniform, bad)


def test_swapped_eps_classes_are_caught():
    def bad(la, eps):
        c = oracle.eps_class(la, eps)
        return np.where(c == 0, 2, np.where(c == 2, 0, c))
    _fails(pins.pin_eps_classes, bad)


def test_strict_eps_threshold_is_caught():
    def bad(la, eps):
        out = np.full(la.shape, -1, np.int8)
        ok = ~np.isnan(la)
        A = np.exp(la[ok])
        out[ok] = np.where(A < eps, 0, np.where(A > 1 - eps, 2, 1))
        return out
    _fails(pins.pin_eps_classes, bad)


def test_carry_taking_root_rows_one_position_short_is_caught():
    def bad(layout, state_seg, row_vals, prev):
        out = oracle.carry_state(layout, state_seg, row_vals, prev)
        for k in ("lp0",):
            v = out[k]
            v[:, 1:] = v[:, :-1].copy()                # every value one position late
        return out
    _fails(pins.pin_carry_example5, bad)


def test_carry_ignoring_the_reached_state_is_caught():
    def bad(layout, state_seg, row_vals, prev):
        roots = np.asarray(layout.chain_seg0[:-1], dtype=state_seg.dtype)
        return oracle.carry_state(layout, roots, row_vals, prev)   # as if all rejected
    _fails(pins.pin_carry_example5, bad)


def test_bfs_expanding_infeasible_requests_is_caught():
    def bad(T, n_pf, depth_cap, cuts):
        # every request treated as feasible: no deferral (Condition 1 dropped)
        from collections import deque
        acc, rej, req, node_cut, deferred = [-1], [-1], [-1], [T], [-1]
        seg_cut, seg_src, seg_of = [T], [-1], [0]
        q, k = deque([0]), 0
        while q and len(seg_cut) - 1 < n_pf and k < len(cuts):
            v = q.popleft()
            c = int(cuts[k])
            k += 1
            s = len(seg_cut)
            seg_cut.append(c)
            seg_src.append(seg_of[v])
            a, b = len(acc), len(acc) + 1
            for _ in range(2):
                acc.append(-1), rej.append(-1), req.append(-1), deferred.append(-1)
            node_cut += [c, node_cut[v]]
            seg_of += [s, seg_of[v]]
            acc[v], rej[v], req[v] = a, b, s
            q += [a, b]
        seg_cut[0] = min(seg_cut[1:]) if len(seg_cut) > 1 else T
        return dict(acc=acc, rej=rej, req=req, node_cut=node_cut, deferred=deferred,
                    seg_cut=seg_cut, seg_src=seg_src)
    _fails(pins.pin_bfs_condition1, bad)


def test_bfs_rejection_child_taking_the_cut_is_caught():
    def bad(T, n_pf, depth_cap, cuts):
        t = OT.bfs(T, n_pf, depth_cap, cuts)
        t = {k: list(v) if hasattr(v, "__len__") else v for k, v in t.items()}
        for v in range(len(t["acc"])):
            r = t["req"][v]
            if r >= 0 and t["rej"][v] >= 0:
                t["node_cut"][t["rej"][v]] = t["seg_cut"][r]
        return t
    _fails(pins.pin_bfs_condition1, bad)


def test_dp_with_swapped_branch_probabilities_is_caught():
    def bad(acc, rej, cand, h, budget):
        return OT.allocation_dp(acc, rej, cand, 1.0 - np.asarray(h), budget)
    _fails(pins.pin_dp_brute_force, bad, OT.allocation_brute, OT.reaching_weights)


def test_dp_spending_the_whole_budget_below_is_caught():
    def bad(acc, rej, cand, h, budget):
        # V(v, b) = 1 + max_m {h V(v+, m) + (1-h) V(v-, b - m)}: the node itself not paid for
        acc = [int(a) for a in acc]
        rej = [int(r) for r in rej]
        from functools import lru_cache

        @lru_cache(maxsize=None)
        def V(v, b):
            if v < 0 or b == 0 or not cand[v]:
                return 0.0
            return 1.0 + max(h[v] * V(acc[v], m) + (1 - h[v]) * V(rej[v], b - m)
                             for m in range(b + 1))
        val = V(0, budget)
        return val, np.zeros(len(acc), bool)
    _fails(pins.pin_dp_brute_force, bad, OT.allocation_brute, OT.reaching_weights)
