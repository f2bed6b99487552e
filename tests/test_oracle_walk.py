"""Pins for the oracle's walk (section 3.2 step (3)), its sequential replay
(Proposition 1) and the expected transition count (Lemma 1)."""

import itertools
import math

import numpy as np

import oracle
from synth import make_workload
from synth.trees import DEFERRED, assemble_layout, bfs_tree
from tests import pins
from tests.helpers import logits_np


def test_example5_path():
    pins.pin_example5(oracle.walk)


def _small_trees(rng, n):
    out = []
    while len(out) < n:
        t = bfs_tree(rng, int(rng.integers(2, 10)), int(rng.integers(1, 9)))
        if t.n_requests >= 1:
            out.append(t)
    return out


def test_brute_force_all_decision_patterns():
    # every accept/reject pattern over the requests of small trees: the walk
    # must follow the pattern (u = A/2 accepts, u = (1+A)/2 rejects), count one
    # transition per scored decision and end in the last accepted state
    rng = np.random.default_rng(31)
    for t in _small_trees(rng, 25):
        lay = assemble_layout([t])
        nreq = lay.n_seg - 1
        logA = np.concatenate([[np.nan], np.log(rng.uniform(0.05, 0.95, nreq))])
        A = np.exp(logA)
        for bits in itertools.product((0, 1), repeat=nreq):
            u = np.ones(lay.n_seg)
            for s in range(1, lay.n_seg):
                u[s] = A[s] / 2 if bits[s - 1] else (1 + A[s]) / 2
            out = oracle.walk(lay, logA, u, max_steps=100)
            v, state, path = 0, 0, [0]
            while lay.req[v] >= 0:
                s = int(lay.req[v])
                if bits[s - 1]:
                    v, state = int(lay.acc[v]), s
                else:
                    v = int(lay.rej[v])
                path.append(v)
            assert out["path"][0] == path
            assert int(out["k_delta"][0]) == len(path) - 1
            assert int(out["state_seg"][0]) == state
            assert int(out["end_node"][0]) == v


def test_walk_stops_at_deferred_node_and_at_max_steps():
    rng = np.random.default_rng(32)
    seen_deferred = 0
    for t in _small_trees(rng, 60):
        lay = assemble_layout([t])
        logA = np.zeros(lay.n_seg)            # A = 1: always accept
        u = np.ones(lay.n_seg)
        out = oracle.walk(lay, logA, u, max_steps=100)
        end = int(out["end_node"][0])
        assert lay.req[end] < 0               # a leaf or a deferred node
        seen_deferred += int(lay.req[end] == DEFERRED)
        for m in range(0, 4):
            o2 = oracle.walk(lay, logA, u, max_steps=m)
            assert int(o2["k_delta"][0]) == min(m, int(out["k_delta"][0]))
            assert o2["path"][0] == out["path"][0][:int(o2["k_delta"][0]) + 1]
    assert seen_deferred > 0


def test_nan_log_accept_rejects():
    lay = assemble_layout([bfs_tree(np.random.default_rng(3), 8, 1)])
    out = oracle.walk(lay, np.array([np.nan, np.nan]), np.array([1.0, 1e-300]), 10)
    assert int(out["k_delta"][0]) == 1 and int(out["state_seg"][0]) == 0


def test_sequential_replay_matches_walk():
    # Proposition 1: with shared random inputs, the walk's state after every
    # transition equals sequential PowerMH's
    for seed in range(6):
        w = make_workload(1, seed=500 + seed, n_pf=8, depth_cap=6, max_steps=6)
        lg, dt = logits_np(w.logits)
        res = oracle.score_subtree(lg, dt, w.V, w.tokens.numpy(), w.layout, w.alpha, w.tau)
        # also make some decisions uncertain so both branches occur
        out = oracle.walk(w.layout, res["log_accept"], w.u, w.max_steps)
        seq = oracle.replay(w.layout, res["lp0"], res["lq"], w.alpha, w.u, w.max_steps)
        st = oracle.materialize(w.layout, 0)
        path = out["path"][0]
        assert len(seq[0]) == len(path)
        for k, v in enumerate(path):
            assert np.array_equal(seq[0][k], st.rows[v])


def test_monte_carlo_transition_count_matches_lemma1():
    # Lemma 1: E[k_Delta] = sum over visited-able decision nodes of R(v)
    rng = np.random.default_rng(33)
    for t in _small_trees(rng, 4):
        lay = assemble_layout([t])
        logA = np.concatenate([[np.nan], np.log(rng.uniform(0.02, 1.0, lay.n_seg - 1))])
        for m in (2, 100):
            want = float(oracle.expected_transitions(lay, logA, m)[0])
            n = 20000
            ks = np.empty(n)
            for i in range(n):
                u = 1.0 - rng.random(lay.n_seg)
                ks[i] = oracle.walk(lay, logA, u, m)["k_delta"][0]
            se = ks.std() / math.sqrt(n) + 1e-12
            assert abs(ks.mean() - want) <= 4 * se + 1e-9, (ks.mean(), want, se)


def test_eps_certain_fraction():
    la = np.log(np.array([1.0, 0.995, 0.5, 0.0099, 0.009, 1e-9]))
    assert oracle.eps_certain_fraction(la, 0.01) == 5 / 6
