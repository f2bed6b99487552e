"""The seeded generator: BFS follows the pages' Example 2; draws are reproducible."""

import json
import os

import numpy as np
import torch

from synth import make_workload
from synth.trees import DEFERRED, LEAF, assemble_layout, bfs_tree

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


class _Scripted:
    """An rng stand-in that returns scripted cuts."""

    def __init__(self, cuts):
        self.cuts = list(cuts)

    def integers(self, lo, hi):
        c = self.cuts.pop(0)
        assert lo <= c < hi
        return c


def test_example2_bfs_order():
    with open(os.path.join(GOLDEN, "example2_bfs.json")) as fh:
        g = json.load(fh)
    T, c1, c2 = 20, 11, 6
    t = bfs_tree(_Scripted([c1, c2]), T, g["n_pf"])
    assert t.n_requests == 2
    # requests at v1 = acc(v0) and v3 = acc(v1), in that order
    assert t.acc[0] == 1 and t.rej[0] == 2 and t.acc[1] == 3 and t.rej[1] == 4
    assert t.req[0] == 1 and t.req[1] == 2 and t.req[2] == LEAF
    assert t.seg_cut[1:] == [c1, c2] and t.seg_src[1:] == [0, 1]
    assert t.node_cut[0] == T and t.node_cut[2] == T and t.node_cut[4] == c1


def test_infeasible_request_is_deferred_and_rejection_child_enqueued():
    T, c1 = 20, 5
    # v1 draws 9 > c1 (deferred); BFS then expands v2 (cut T) and v4 (cut c1)
    t = bfs_tree(_Scripted([c1, 9, 13, 2]), T, 3)
    assert t.req[1] == DEFERRED and t.deferred_cut[1] == 9
    assert t.req[2] == 2 and t.seg_cut[2] == 13          # v2: rejection child of v0
    assert t.req[4] == 3 and t.seg_cut[3] == 2 and t.node_cut[4] == c1
    assert t.seg_src[3] == 1                             # v4 keeps v1's state y


def test_workloads_are_reproducible():
    a = make_workload(1)
    b = make_workload(1)
    assert torch.equal(a.logits, b.logits) and torch.equal(a.tokens, b.tokens)
    assert np.array_equal(a.u, b.u)
    assert np.array_equal(a.layout.seg_cut, b.layout.seg_cut)
    assert a.layout.n_rows == a.logits.shape[0]
    assert (a.u > 0).all() and (a.u <= 1).all()


def test_multi_chain_layout_offsets():
    rng = np.random.default_rng(7)
    ts = [bfs_tree(rng, 16, 4) for _ in range(5)]
    lay = assemble_layout(ts)
    assert lay.n_chains == 5
    for c in range(5):
        s0, s1 = lay.chain_seg0[c], lay.chain_seg0[c + 1]
        assert lay.seg_src[s0] == -1
        for s in range(s0 + 1, s1):
            assert s0 <= lay.seg_src[s] < s1
        assert np.all(np.diff(lay.seg_row0[s0:s1 + 1]) == 16 - lay.seg_cut[s0:s1])
