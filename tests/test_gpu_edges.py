"""GPU parity on degenerate and extreme batches: chains without requests,
a batch without rows, one-row segments, a 2^20-token vocabulary and many
small chains in one launch."""

import numpy as np
import pytest
import torch

from synth.trees import assemble_layout, bfs_tree
from synth.workload import Workload, draw_tokens, gen_logits
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _workload(trees, V, dtype="bf16", tau=0.25, alpha=4.0, seed=0, ld=None, max_steps=50):
    rng = np.random.default_rng(seed)
    lay = assemble_layout(trees)
    ldv = V if ld is None else ld
    n = lay.n_rows
    if n:
        x = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), n, V, dtype, seed=seed + 1,
                       device=DEV)
        if ldv != V:
            big = torch.full((n, ldv), float("nan"), dtype=x.dtype, device=DEV)
            big[:, :V] = x
            x = big
        tok = draw_tokens(x, tau, seed=seed + 2, V=V)
    else:
        x = torch.empty((0, ldv), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                        device=DEV)
        tok = torch.empty(0, dtype=torch.int32, device=DEV)
    return Workload(name="edge", layout=lay, V=V, dtype=dtype, alpha=alpha, tau=tau, logits=x,
                    tokens=tok, u=1.0 - rng.random(lay.n_seg), max_steps=max_steps)


def test_chains_without_requests_next_to_normal_chains():
    rng = np.random.default_rng(61)
    trees = []
    for i in range(12):
        trees.append(bfs_tree(rng, 16, 0 if i % 3 == 0 else 4))
    w = _workload(trees, 4096, seed=61)
    s = H.full_parity(w)
    g = H.run_gpu(w)
    lay = w.layout
    for c in range(0, 12, 3):                 # a root alone: no transition, state = root
        assert g["k_delta"][c] == 0
        assert g["state_seg"][c] == lay.chain_seg0[c]
    assert s["lp0_max_rel"] <= H.TOK_RTOL


def test_batch_without_rows():
    rng = np.random.default_rng(62)
    trees = [bfs_tree(rng, 8, 0) for _ in range(5)]
    w = _workload(trees, 1000, dtype="f32", seed=62)
    assert w.n_rows == 0
    g = H.run_gpu(w)
    assert g["status"] == 0 and g["wstatus"] == 0
    assert np.isnan(g["log_accept"]).all()
    assert (g["k_delta"] == 0).all()
    assert np.array_equal(g["state_seg"], w.layout.chain_seg0[:-1])


def test_one_row_segments():
    # T = 1: every suffix is the single position 1
    rng = np.random.default_rng(63)
    trees = [bfs_tree(rng, 1, 3) for _ in range(20)]
    w = _workload(trees, 2048, seed=63)
    assert w.n_rows == sum(t.suffix_tokens() + (1 - t.seg_cut[0]) for t in trees)
    H.full_parity(w)


@pytest.mark.parametrize("V,ld", [(1 << 20, None), ((1 << 20) + 24, (1 << 20) + 32)])
def test_two_million_byte_rows(V, ld):
    # rows of 2 MB: each row spans hundreds of chunks and many warps, so every
    # row's result is merged from partials
    rng = np.random.default_rng(64)
    w = _workload([bfs_tree(rng, 4, 2)], V, seed=64, ld=ld)
    H.full_parity(w)


def test_many_small_chains_in_one_launch():
    rng = np.random.default_rng(65)
    trees = [bfs_tree(rng, int(rng.integers(1, 24)), int(rng.integers(0, 6)))
             for _ in range(1)]
    T = trees[0].T
    trees += [bfs_tree(rng, T, int(rng.integers(0, 6))) for _ in range(1999)]
    w = _workload(trees, 512, dtype="f32", seed=65)
    H.full_parity(w)


def test_bad_uniform_is_flagged_and_rejects():
    # u outside (0, 1] is reported (PS_DEV_BAD_UNIFORM) and that decision rejects
    rng = np.random.default_rng(66)
    w = _workload([bfs_tree(rng, 16, 4) for _ in range(3)], 2048, seed=66)
    lay = w.layout
    s_bad = int(lay.req[int(lay.chain_node0[1])])      # the first decision of chain 1
    u = w.u.copy()
    u[s_bad] = 0.0
    w.u = u
    g = H.run_gpu(w)
    assert g["wstatus"] & 0x80
    root1 = int(lay.chain_node0[1])
    assert g["path"][1 * (w.max_steps + 1) + 1] == int(lay.rej[root1])   # went right


def test_request_whose_src_is_in_another_chain_is_flagged():
    # a layout the host validator would reject, given to the device anyway:
    # the request gets NaN and PS_DEV_BAD_LAYOUT, the others are unaffected
    rng = np.random.default_rng(67)
    w = _workload([bfs_tree(rng, 16, 4) for _ in range(2)], 2048, seed=67)
    lay = w.layout
    bad = int(lay.chain_seg0[1]) + 1                    # first request of chain 1
    lay.seg_src = lay.seg_src.copy()
    lay.seg_src[bad] = 1                                # a request of chain 0
    g = H.run_gpu(w)
    assert g["status"] & 0x10
    assert np.isnan(g["log_accept"][bad])
    ok = ~lay.is_root()
    ok[bad] = False
    assert np.isfinite(g["log_accept"][ok]).all()


def test_carry_with_a_foreign_state_is_flagged():
    import mh_prefetch_subtree_gb300 as ps
    rng = np.random.default_rng(68)
    w = _workload([bfs_tree(rng, 16, 4) for _ in range(2)], 2048, seed=68)
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens, V=w.V,
                                alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    d.step()
    torch.cuda.synchronize()
    d.t["state_seg"][1] = 1                             # chain 1 "reached" chain 0's segment
    T = w.layout.T
    prev = {k: torch.zeros((2, T), dtype=torch.float64, device=DEV) for k in ("lp0", "lq")}
    out = d.carry(prev)
    torch.cuda.synchronize()
    assert int(out["status"].item()) & 0x10
    assert torch.isnan(out["lp0"][1]).all() and torch.isfinite(out["lp0"][0]).all()


def test_chain_larger_than_the_walks_shared_memory_stage():
    # one chain of 300 requests: 1,669 nodes and 301 segments, more than the
    # walk stages in shared memory (512 nodes, 256 segments), so it walks from
    # global memory; against the oracle through the one-call round, and the
    # walk kernel of ps_walk_subtree gives the same path
    import mh_prefetch_subtree_gb300 as ps
    rng = np.random.default_rng(69)
    w = _workload([bfs_tree(rng, 64, 300)], 1024, dtype="f32", seed=69, max_steps=100)
    lay = w.layout
    assert len(lay.acc) > 512 and lay.n_seg > 256
    s = H.full_parity(w)
    d = ps.DeviceSubtree.create(layout=lay, u=w.u, logits=w.logits, tokens=w.tokens, V=w.V,
                                alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    d.step(fused=False)
    torch.cuda.synchronize()
    g = H.run_gpu(w)
    for k in ("state_seg", "end_node", "k_delta", "path"):
        assert np.array_equal(d.t[k].cpu().numpy(), g[k]), k
    assert s["k_delta_mean"] >= 1
