"""Pins for the oracle's per-token log-probabilities (CPU only).

What the pages fix: log p0 and log q_tau of the sampled token come from the
same logits without and with temperature scaling (PreSTO Appendix B.1, last
paragraph; Appendix D.3).  The pins below are closed forms, special cases and
a library routine, chosen so that a dropped term, a wrong temperature, a wrong
token index or an inaccurate log1p fails one of them.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import bf16_from_float, float_from_bf16


def _rows(x, dtype):
    x = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_from_float(x)
    return x


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 2, 7, 1024, 4099])
def test_uniform_row_is_minus_log_V(dtype, V):
    # all logits equal => softmax is uniform at every temperature
    rng = np.random.default_rng(V)
    n = 5
    val = rng.normal(size=(n, 1)).astype(np.float32)
    x = np.repeat(val, V, axis=1)
    tok = rng.integers(0, V, n).astype(np.int32)
    for tau in (0.25, 1.0, 0.37):
        lp0, lq = oracle.row_logprobs(_rows(x, dtype), dtype, V, tok, tau)
        np.testing.assert_allclose(lp0, -math.log(V), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(lq, -math.log(V), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_tau_one_gives_identical_log_probs(dtype):
    rng = np.random.default_rng(1)
    x = rng.normal(scale=3.0, size=(20, 333)).astype(np.float32)
    tok = rng.integers(0, 333, 20).astype(np.int32)
    lp0, lq = oracle.row_logprobs(_rows(x, dtype), dtype, 333, tok, 1.0)
    assert np.array_equal(lp0, lq)


@pytest.mark.parametrize("tau", [0.25, 0.125, 0.7, 1.0, 2.0])
def test_two_token_closed_form(tau):
    # V = 2: log p(tok) = log sigmoid((l_tok - l_other) / tau)
    rng = np.random.default_rng(2)
    x = rng.normal(scale=4.0, size=(50, 2)).astype(np.float32)
    tok = rng.integers(0, 2, 50).astype(np.int32)
    lp0, lq = oracle.row_logprobs(x, "f32", 2, tok, tau)
    d = (x[np.arange(50), tok].astype(np.float64)
         - x[np.arange(50), 1 - tok].astype(np.float64))
    np.testing.assert_allclose(lp0, -np.logaddexp(0.0, -d), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(lq, -np.logaddexp(0.0, -d / tau), rtol=1e-13, atol=1e-300)


def test_single_token_vocab_is_zero():
    x = np.array([[3.5], [-100.0], [0.0]], dtype=np.float32)
    lp0, lq = oracle.row_logprobs(x, "f32", 1, np.zeros(3, np.int32), 0.25)
    assert np.all(lp0 == 0.0) and np.all(lq == 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tau", [0.25, 0.5, 1.0, 0.3])
def test_matches_torch_log_softmax(dtype, tau):
    # library routine: torch.log_softmax in float64 on the CPU
    rng = np.random.default_rng(3)
    V = 517
    x = (rng.normal(scale=3.0, size=(40, V))).astype(np.float32)
    x[:, 7] += 9.0                      # a peaked column
    x[3, :] = -np.inf
    x[3, 11] = 1.0                      # masked vocabulary: a single finite logit
    x[4, 100:] = -np.inf
    tok = rng.integers(0, V, 40).astype(np.int32)
    tok[3] = 11
    tok[4] = 50
    stored = _rows(x, dtype)
    vals = float_from_bf16(stored) if dtype == "bf16" else stored
    lp0, lq = oracle.row_logprobs(stored, dtype, V, tok, tau)
    t = torch.from_numpy(vals.astype(np.float64))
    ref0 = torch.log_softmax(t, dim=1)[torch.arange(40), torch.from_numpy(tok).long()]
    refq = torch.log_softmax(t / tau, dim=1)[torch.arange(40), torch.from_numpy(tok).long()]
    np.testing.assert_allclose(lp0, ref0.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lq, refq.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("V", [2, 1024, 151936])
def test_dominant_token_keeps_relative_accuracy(V):
    # a single logit 30 above all others (which are 0): closed forms
    #   lp0 = -log1p((V-1) e^-30),  lq = -log1p((V-1) e^(-30/tau))
    # the second is ~1e-50 for tau = 0.25 and needs log1p of the excluded sum;
    # rtol covers the float64 rounding of a sequential sum of V-1 equal terms
    x = np.zeros((1, V), dtype=np.float32)
    x[0, V // 3] = 30.0
    tok = np.array([V // 3], np.int32)
    for dtype in ("bf16", "f32"):
        lp0, lq = oracle.row_logprobs(_rows(x, dtype), dtype, V, tok, 0.25)
        np.testing.assert_allclose(lp0[0], -math.log1p((V - 1) * math.exp(-30.0)), rtol=1e-10)
        np.testing.assert_allclose(lq[0], -math.log1p((V - 1) * math.exp(-120.0)), rtol=1e-10)
        assert lq[0] < 0.0


def test_row_index_and_ld():
    rng = np.random.default_rng(4)
    V, ld = 100, 112
    pool = rng.normal(size=(9, ld)).astype(np.float32)
    idx = np.array([3, 3, 0, 8, 5], np.int64)
    tok = rng.integers(0, V, 5).astype(np.int32)
    a0, aq = oracle.row_logprobs(pool, "f32", V, tok, 0.25, row_index=idx)
    b0, bq = oracle.row_logprobs(np.ascontiguousarray(pool[idx, :V]), "f32", V, tok, 0.25)
    assert np.array_equal(a0, b0) and np.array_equal(aq, bq)


def test_invalid_rows_give_nan():
    x = np.zeros((3, 4), dtype=np.float32)
    x[1, 2] = np.nan
    x[2, :] = -np.inf
    tok = np.array([4, 0, 0], np.int32)     # row 0: token out of range
    lp0, lq = oracle.row_logprobs(x, "f32", 4, tok, 0.5)
    assert np.isnan(lp0).all() and np.isnan(lq).all()


def test_threads_do_not_change_results():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(64, 300)).astype(np.float32)
    tok = rng.integers(0, 300, 64).astype(np.int32)
    a = oracle.row_logprobs(x, "f32", 300, tok, 0.25, threads=1)
    b = oracle.row_logprobs(x, "f32", 300, tok, 0.25, threads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
