"""Host logic of bench.py that needs no GPU: the bounded samples on which the
reference arm times the oracle.

A sample must be a subtree batch of its own (every kept request proposes from
a kept segment and satisfies Condition 1 of the PreSTO pages, section 3.2, and
the root's rows cover every position a kept request's x suffix reads), and it
must stay within the row budget it was given wherever the tree allows.
"""

import copy
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth.trees import LEAF, assemble_layout  # noqa: E402
from synth.workload import CONFIGS, _trees_for  # noqa: E402


def _tree(cfg_id):
    cfg = dict(CONFIGS[cfg_id])
    return _trees_for(cfg, np.random.default_rng(10086 + cfg_id))[0]


def _check_batch(t):
    T = t.T
    n = len(t.seg_cut)
    assert n >= 2, "a sample holds at least one request"
    assert t.seg_src[0] == -1
    for i in range(1, n):
        src = t.seg_src[i]
        assert 0 <= src < i
        c_src = T if src == 0 else t.seg_cut[src]
        assert t.seg_cut[i] <= c_src                          # Condition 1
        assert t.seg_cut[0] <= t.seg_cut[i] <= T - 1          # root rows cover c_i+1..c_src
    for r in t.req:
        assert r < n and (r >= 0 or r in (LEAF, -2))
    lay = assemble_layout([t])
    assert lay.n_rows == sum(T - c for c in t.seg_cut)
    return lay


@pytest.mark.parametrize("cfg_id", [2, 3, 4])
def test_short_runs_keep_the_root_and_the_first_requests(cfg_id):
    full = _tree(cfg_id)
    t = bench.reference_sample_tree(copy.deepcopy(full), 90 * 7000 // 5)
    lay = _check_batch(t)
    root_rows = full.T - full.seg_cut[0]
    assert t.seg_cut[0] == full.seg_cut[0]
    assert t.seg_cut[1:] == full.seg_cut[1:len(t.seg_cut)]
    req_rows = lay.n_rows - root_rows
    assert req_rows <= 2500 or len(t.seg_cut) == 2


@pytest.mark.parametrize("cfg_id", [2, 3, 4])
@pytest.mark.parametrize("steps", [200, 510, 2010])
def test_long_runs_keep_one_request_from_the_root(cfg_id, steps):
    full = _tree(cfg_id)
    budget = 90 * 7000 // steps
    root_rows = full.T - full.seg_cut[0]
    if root_rows + full.T - full.seg_cut[1] <= budget:
        pytest.skip("the root and the first request fit this budget")
    t = bench.reference_sample_tree(copy.deepcopy(full), budget)
    lay = _check_batch(t)
    assert len(t.seg_cut) == 2 and t.seg_src[1] == 0
    c = t.seg_cut[1]
    assert c in full.seg_cut[1:]                     # a request of the same tree
    assert t.seg_cut[0] == c and lay.n_rows == 2 * (full.T - c)
    fits = [x for x in full.seg_cut[1:] if 2 * (full.T - x) <= budget]
    if fits:
        assert c == min(fits) and lay.n_rows <= budget   # the longest suffix that fits
    else:
        assert c == max(full.seg_cut[1:])                # else the shortest one
    # the walk from the root reaches the one request's decision
    assert t.req[0] == 1 and t.acc[0] >= 0 and t.rej[0] >= 0


def test_sample_budget_shrinks_with_the_run():
    full = _tree(3)
    rows = []
    for kw in (5, 60, 200, 510, 2010):
        t = bench.reference_sample_tree(copy.deepcopy(full), 90 * 7000 // kw)
        rows.append(assemble_layout([t]).n_rows)
    assert rows == sorted(rows, reverse=True) and rows[-1] < rows[0]
