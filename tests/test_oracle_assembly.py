"""Pins for the oracle's suffix sums, log A (eq. (6)) and state materialisation."""

import numpy as np

import oracle
from synth import make_workload
from synth.trees import assemble_layout, bfs_tree
from tests import pins
from tests.helpers import logits_np


def test_uniform_rows_give_exact_counts():
    pins.pin_uniform_counts(oracle.row_logprobs, oracle.suffix_sums)


def test_mh_rule_closed_form_tau_one():
    pins.pin_mh_closed_form(oracle.row_logprobs, oracle.suffix_sums, oracle.log_accept)


def test_alpha_tau_one_accepts_everything():
    pins.pin_alpha_tau_one(oracle.row_logprobs, oracle.suffix_sums, oracle.log_accept)


def test_copied_suffix_gives_zero():
    pins.pin_y_equals_x(oracle.row_logprobs, oracle.suffix_sums, oracle.log_accept,
                        oracle.materialize)


def test_reverse_move_is_antisymmetric():
    pins.pin_reversal(oracle.row_logprobs, oracle.suffix_sums, oracle.log_accept)


def test_two_segment_rule_matches_materialisation():
    pins.pin_two_segment_rule(oracle.materialize)


def test_rejection_child_inherits_state():
    pins.pin_rejection_inherits(oracle.materialize)


def test_sum_of_segments_is_sum_of_whole():
    # brute force: the x-sum of a request equals the per-position sum over
    # the explicit from-state, accumulated one position at a time
    w = make_workload(1)
    lg, dt = logits_np(w.logits)
    res = oracle.score_subtree(lg, dt, w.V, w.tokens.numpy(), w.layout, w.alpha, w.tau)
    st = oracle.materialize(w.layout, 0)
    for v in range(w.layout.n_nodes):
        s = int(w.layout.req[v])
        if s < 0:
            continue
        c = int(w.layout.seg_cut[s])
        acc = 0.0
        for t in range(c + 1, w.layout.T + 1):
            acc += res["lp0"][st.rows[v][t]]
        np.testing.assert_allclose(res["lp_x"][s], acc, rtol=1e-12)


def test_condition1_holds_for_generated_trees():
    rng = np.random.default_rng(21)
    for _ in range(200):
        T = int(rng.integers(1, 64))
        t = bfs_tree(rng, T, int(rng.integers(1, 20)), None)
        lay = assemble_layout([t])
        for s in range(1, lay.n_seg):
            src = int(lay.seg_src[s])
            csrc = T if src == 0 else int(lay.seg_cut[src])
            assert 0 <= lay.seg_cut[s] <= csrc
        # every deferred draw really was infeasible under its node's cut
        for v, c in t.deferred_cut.items():
            assert c > t.node_cut[v]


def test_config1_end_to_end_is_finite_and_reproducible():
    w = make_workload(1)
    lg, dt = logits_np(w.logits)
    a = oracle.score_subtree(lg, dt, w.V, w.tokens.numpy(), w.layout, w.alpha, w.tau)
    b = oracle.score_subtree(lg, dt, w.V, w.tokens.numpy(), w.layout, w.alpha, w.tau,
                             threads=1)
    req = ~w.layout.is_root()
    assert np.isfinite(a["log_accept"][req]).all()
    assert (a["log_accept"][req] <= 0).all()
    for k in ("lp0", "lq", "log_accept"):
        assert np.array_equal(a[k], b[k], equal_nan=True)
