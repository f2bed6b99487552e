"""Trees built by libps's own host BFS (ps_build_bfs_tree) feed the GPU
scoring and walk, checked against the oracle: the host construction and the
device path agree on one layout, deferred stops included."""

from types import SimpleNamespace

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth.trees import assemble_layout
from synth.workload import Workload, draw_tokens, gen_logits
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _libps_tree(rng, T, n_pf, depth_cap=None):
    cuts = rng.integers(0, T, 6 * n_pf + 4).astype(np.int32)
    g = ps.ps_build_bfs_tree(T, n_pf, depth_cap, cuts)
    return SimpleNamespace(T=T, acc=list(g["acc"]), rej=list(g["rej"]), req=list(g["req"]),
                           seg_cut=list(g["seg_cut"]), seg_src=list(g["seg_src"]),
                           deferred_cut=list(g["deferred_cut"]))


@pytest.mark.parametrize("T,n_pf,chains,cap", [(64, 8, 6, 4), (512, 16, 3, None),
                                               (1024, 16, 1, None)])
def test_host_bfs_trees_through_the_device_path(T, n_pf, chains, cap):
    rng = np.random.default_rng(T + n_pf)
    trees = [_libps_tree(rng, T, n_pf, cap) for _ in range(chains)]
    lay = assemble_layout(trees)
    V = 151936 if T >= 512 else 4096
    x = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), lay.n_rows, V, "bf16",
                   seed=T, device=DEV)
    tok = draw_tokens(x, 0.25, seed=T + 1)
    w = Workload(name="libps bfs", layout=lay, V=V, dtype="bf16", alpha=4.0, tau=0.25,
                 logits=x, tokens=tok, u=1.0 - rng.random(lay.n_seg), max_steps=100)
    s = H.full_parity(w)
    # a walk that ends at a deferred node ends where the host recorded a cut
    g = H.run_gpu(w)
    for c in range(chains):
        end = int(g["end_node"][c]) - int(lay.chain_node0[c])
        t = trees[c]
        if t.req[end] == ps.PS_NODE_DEFERRED:
            assert 0 <= t.deferred_cut[end] < T
    assert s["lp0_max_rel"] <= H.TOK_RTOL
