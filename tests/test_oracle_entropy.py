"""Pins for the oracle's by-products: entropy of p0 per row (PreSTO Appendix
D.3, quantity (iii)) and the epsilon-certainty class of each decision
(section 3.3)."""

import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import bf16_from_float, float_from_bf16


def _ent(x, dtype="f32", tau=0.25):
    V = x.shape[1]
    stored = bf16_from_float(x) if dtype == "bf16" else x.astype(np.float32)
    tok = np.zeros(x.shape[0], np.int32)
    return oracle.row_logprobs(stored, dtype, V, tok, tau, entropy=True)[2], stored


@pytest.mark.parametrize("V", [1, 2, 9, 1024, 151936])
def test_uniform_row_entropy_is_log_V(V):
    h, _ = _ent(np.full((3, V), 1.25, np.float32))
    np.testing.assert_allclose(h, math.log(V), rtol=1e-12, atol=1e-15)


def test_two_token_closed_form():
    rng = np.random.default_rng(1)
    x = rng.normal(scale=4.0, size=(40, 2)).astype(np.float32)
    h, _ = _ent(x)
    d = x[:, 0].astype(np.float64) - x[:, 1]
    p = 1.0 / (1.0 + np.exp(-d))
    want = -(p * np.log(p) + (1 - p) * np.log1p(-p))
    np.testing.assert_allclose(h, want, rtol=1e-10, atol=1e-14)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_matches_torch_categorical_entropy(dtype):
    # library routine: torch.distributions.Categorical in float64
    rng = np.random.default_rng(2)
    x = rng.normal(scale=3.0, size=(30, 700)).astype(np.float32)
    x[:, 3] += 10.0
    x[5, 100:] = -np.inf
    h, stored = _ent(x, dtype)
    vals = float_from_bf16(stored) if dtype == "bf16" else stored
    want = torch.distributions.Categorical(logits=torch.from_numpy(vals.astype(np.float64))).entropy()
    np.testing.assert_allclose(h, want.numpy(), rtol=1e-11, atol=1e-13)


def test_peaked_row_closed_form():
    # one logit 30 above V-1 zeros: p_big = 1/(1+k), k = (V-1) e^-30, and
    # H = log(1 + k) + 30 k / (1 + k)
    V = 5000
    x = np.zeros((1, V), np.float32)
    x[0, 17] = 30.0
    h, _ = _ent(x)
    k = (V - 1) * math.exp(-30.0)
    np.testing.assert_allclose(h[0], math.log1p(k) + 30.0 * k / (1.0 + k), rtol=1e-9)


def test_entropy_does_not_depend_on_the_token_or_tau():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(4, 300)).astype(np.float32)
    a = oracle.row_logprobs(x, "f32", 300, np.array([0, 1, 2, 3], np.int32), 0.25, entropy=True)[2]
    b = oracle.row_logprobs(x, "f32", 300, np.array([9, 8, 7, 6], np.int32), 1.0, entropy=True)[2]
    assert np.array_equal(a, b)


def test_eps_classes():
    A = np.array([1.0, 0.995, 0.99, 0.5, 0.0101, 0.0099, 0.0, np.nan])
    with np.errstate(divide="ignore"):
        la = np.log(A)
    cls = oracle.eps_class(la, 0.01)
    assert list(cls) == [2, 2, 2, 1, 1, 0, 0, -1]
    assert oracle.eps_certain_fraction(la[:-1], 0.01) == 5 / 7
