"""ps_score_walk_subtree (one call per round) against ps_score_subtree then
ps_walk_subtree, and masked rows mixed with ordinary ones in the entropy
variant.

The one-call round computes the same suffix sums, log A and walk as the two
calls (PreSTO section 3.2 steps (2)-(3), eq. (6)), in fewer launches; its
outputs must be identical bit for bit.  The other tests run every parity test
through it already (the harness's step is the one-call round); these pin it to
the two-call sequence directly, on layouts with one chain, many chains, chains
without requests and a batch without rows.
"""

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth import make_workload
from synth.trees import assemble_layout, bfs_tree
from synth.workload import Workload, draw_tokens, gen_logits
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
KEYS = ("lp0", "lq", "lp_y", "lq_y", "lp_x", "lq_x", "log_ratio", "log_accept", "entropy",
        "eps_class", "state_seg", "end_node", "k_delta", "path", "status", "wstatus")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _chains(n_chains, T, n_pf, V=4096, seed=0, every_third_empty=False):
    rng = np.random.default_rng(seed)
    trees = [bfs_tree(rng, T, 0 if (every_third_empty and i % 3 == 0) else n_pf)
             for i in range(n_chains)]
    lay = assemble_layout(trees)
    if lay.n_rows:
        x = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), lay.n_rows, V, "bf16",
                       seed=seed + 1, device=DEV)
        tok = draw_tokens(x, 0.25, seed=seed + 2)
    else:
        x = torch.empty((0, V), dtype=torch.bfloat16, device=DEV)
        tok = torch.empty(0, dtype=torch.int32, device=DEV)
    return Workload(name="fused", layout=lay, V=V, dtype="bf16", alpha=4.0, tau=0.25, logits=x,
                    tokens=tok, u=1.0 - rng.random(lay.n_seg), max_steps=100)


def _run(w, fused):
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                row_index=w.row_index, entropy=True, eps=H.EPS)
    for _ in range(2):                       # twice: the chain counters start from zero again
        for k in ("status", "wstatus"):
            d.t[k].zero_()
        d.step(fused=fused)
    torch.cuda.synchronize()
    return {k: d.t[k].cpu().numpy() for k in KEYS if d.t.get(k) is not None}


@pytest.mark.parametrize("case", ["config1", "config2_small", "many_chains", "empty_chains",
                                  "no_rows", "long_segments"])
def test_one_call_round_equals_the_two_calls(case):
    if case == "config1":
        w = make_workload(1, device=DEV)
    elif case == "config2_small":
        w = make_workload(2, device=DEV, T=96, n_pf=10, seed=31)
    elif case == "many_chains":
        w = _chains(300, 24, 6, seed=32)               # 2,100 segments, many waves of blocks
    elif case == "empty_chains":
        w = _chains(12, 16, 4, seed=33, every_third_empty=True)
    elif case == "no_rows":
        w = _chains(5, 8, 0, seed=34)
    else:
        # segments of up to 6000 rows: a request's sums take several rounds of
        # loads per thread
        w = _chains(1, 6000, 6, V=1024, seed=35)
    a = _run(w, fused=True)
    b = _run(w, fused=False)
    assert int(a["status"][0]) == 0 and int(a["wstatus"][0]) == 0, ps.dev_status_names(
        int(a["status"][0]) | int(a["wstatus"][0]))
    for k in b:
        floating = np.issubdtype(b[k].dtype, np.floating)
        assert np.array_equal(a[k], b[k], equal_nan=floating), k
    if w.n_rows:
        H.check_walk(w, a, H.run_oracle(w))


@pytest.mark.parametrize("tau", [0.25, 0.3])
def test_masked_rows_among_ordinary_rows_in_the_entropy_variant(tau):
    # without the masked-logits hint, chunks holding a -inf take the clamped
    # slow path while the other chunks of the same warps stay on the fast
    # path; masked, flat and peaked rows side by side must all match the oracle
    V = 151936
    rng = np.random.default_rng(41)
    trees = [bfs_tree(rng, 40, 6) for _ in range(3)]
    lay = assemble_layout(trees)
    n = lay.n_rows
    x = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), n, V, "bf16", seed=42,
                   device=DEV)
    kind = rng.integers(0, 6, n)
    for r in range(n):
        if kind[r] == 1:
            x[r, 1000:] = float("-inf")                  # masked tail
        elif kind[r] == 2:
            x[r, :50000] = float("-inf")                 # masked head
        elif kind[r] == 3:
            x[r, 20000:120000] = float("-inf")           # masked middle
        elif kind[r] == 4:
            x[r, int(rng.integers(0, V))] = 60.0         # one dominant logit
    tok = draw_tokens(x, tau, seed=43)
    w = Workload(name="masked-mix", layout=lay, V=V, dtype="bf16", alpha=4.0, tau=tau,
                 logits=x, tokens=tok, u=1.0 - rng.random(lay.n_seg), max_steps=100)
    s = H.full_parity(w)
    assert s["lp0_max_rel"] <= H.TOK_RTOL


def test_one_call_round_with_invalid_chain_bounds():
    # the last chain's end in chain_seg0 points past n_seg (a layout the host
    # validator rejects, given to the device anyway): its requests get NaN and
    # PS_DEV_BAD_LAYOUT, it is not walked (its outputs keep their old values),
    # and the other chains are scored and walked as before
    w = _chains(3, 16, 4, seed=36)
    ref = _run(w, fused=True)
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                entropy=True, eps=H.EPS)
    d.t["chain_seg0"][-1] += 5
    for k in ("state_seg", "end_node", "k_delta", "path"):
        d.t[k].fill_(-7)
    d.step()
    torch.cuda.synchronize()
    assert int(d.t["status"].item()) & 0x10
    lay = w.layout
    s2 = int(lay.chain_seg0[2])
    la = d.t["log_accept"].cpu().numpy()
    assert np.isnan(la[s2:]).all()
    assert np.array_equal(la[:s2], ref["log_accept"][:s2], equal_nan=True)
    stride = w.max_steps + 1
    for k in ("state_seg", "end_node", "k_delta"):
        got = d.t[k].cpu().numpy()
        assert np.array_equal(got[:2], ref[k][:2]), k
        assert got[2] == -7, k
    path = d.t["path"].cpu().numpy()
    assert np.array_equal(path[:2 * stride], ref["path"][:2 * stride])
    assert (path[2 * stride:] == -7).all()
