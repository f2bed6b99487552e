"""Planted mistakes in the oracle (on the CPU): each pin must catch its own.

Each test builds a deliberately wrong variant of one oracle function, hands it
to the pin that is meant to catch that kind of mistake, and checks the pin
fails; the unmodified function passes the same pin in the other test files.
"""

import numpy as np
import pytest

import oracle
from tests import pins


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_sign_error_in_log_accept_is_caught():
    def bad(sums, alpha):
        r = (sums["lq_y"] - sums["lq_x"]) + alpha * (sums["lp_x"] - sums["lp_y"])
        return r, np.minimum(0.0, r)
    _fails(pins.pin_mh_closed_form, oracle.row_logprobs, oracle.suffix_sums, bad)


def test_misplaced_alpha_is_caught():
    def bad(sums, alpha):
        r = alpha * (sums["lq_x"] - sums["lq_y"]) + (sums["lp_y"] - sums["lp_x"])
        return r, np.minimum(0.0, r)
    _fails(pins.pin_mh_closed_form, oracle.row_logprobs, oracle.suffix_sums, bad)


def test_missing_clip_is_caught():
    def bad(sums, alpha):
        r = (sums["lq_x"] - sums["lq_y"]) + alpha * (sums["lp_y"] - sums["lp_x"])
        return r, r
    _fails(pins.pin_mh_closed_form, oracle.row_logprobs, oracle.suffix_sums, bad)


def test_off_by_one_suffix_is_caught():
    def bad(layout, lp0, lq, states=None):
        # sums positions c..T-1 instead of c+1..T
        out = {k: np.full(layout.n_seg, np.nan) for k in ("lp_y", "lq_y", "lp_x", "lq_x")}
        st = oracle.materialize(layout, 0)
        for v in range(layout.n_nodes):
            s = int(layout.req[v])
            if s < 0:
                continue
            c = int(layout.seg_cut[s])
            a = int(layout.acc[v])
            y = st.rows[a][max(c, 1):layout.T]
            x = st.rows[v][max(c, 1):layout.T]
            y, x = y[y >= 0], x[x >= 0]
            out["lp_y"][s], out["lq_y"][s] = lp0[y].sum(), lq[y].sum()
            out["lp_x"][s], out["lq_x"][s] = lp0[x].sum(), lq[x].sum()
        return out
    _fails(pins.pin_uniform_counts, oracle.row_logprobs, bad)


def test_rejection_child_taking_the_proposal_is_caught():
    def bad(layout, c):
        st = oracle.materialize(layout, c)
        for v in range(layout.n_nodes):
            a, b = int(layout.acc[v]), int(layout.rej[v])
            if int(layout.req[v]) >= 0 and b >= 0:
                st.rows[b] = st.rows[a]
        return st
    _fails(pins.pin_rejection_inherits, bad)


def test_swapped_children_in_walk_are_caught():
    def bad(layout, logA, u, max_steps):
        class Swapped:
            pass
        sw = Swapped()
        sw.__dict__.update(layout.__dict__)
        sw.acc, sw.rej = layout.rej, layout.acc
        return oracle.walk(sw, logA, u, max_steps)
    _fails(pins.pin_example5, bad)


def test_dropped_temperature_is_caught():
    def bad(logits, dtype, V, tokens, tau, row_index=None, threads=None):
        lp0, _ = oracle.row_logprobs(logits, dtype, V, tokens, tau, row_index, threads)
        return lp0, lp0.copy()
    _fails(pins.pin_library_log_softmax, bad)


def test_naive_log_of_full_sum_is_caught():
    def bad(logits, dtype, V, tokens, tau, row_index=None, threads=None):
        x = logits[:, :V].astype(np.float64)
        m = x.max(axis=1, keepdims=True)
        i = np.arange(x.shape[0])
        lp0 = (x[i, tokens] - m[:, 0]) - np.log(np.exp(x - m).sum(1))
        lq = (x[i, tokens] - m[:, 0]) / tau - np.log(np.exp((x - m) / tau).sum(1))
        return lp0, lq
    _fails(pins.pin_dominant_token, bad)


def test_unmodified_oracle_passes_the_extra_pins():
    pins.pin_library_log_softmax(oracle.row_logprobs)
    pins.pin_dominant_token(oracle.row_logprobs)
