"""ps_score_subtree_noalloc against ps_score_subtree (GPU, through the C ABI).

The no-allocation entry point serves callers that cannot call cudaMalloc (for
instance a hook inside another engine whose device memory belongs to that
engine's pool): it takes no workspace and uses a static device array inside
libps instead.  This file is collected last so that a run stopping at the
first failure has already run every other test; it also builds the library
itself, so it passes when run alone in a fresh process.
"""

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth import make_workload
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _outputs(n_rows, n_seg, per_row):
    f64 = lambda n: torch.full((n,), float("nan"), dtype=torch.float64, device=DEV)
    t = dict(log_accept=f64(n_seg), log_ratio=f64(n_seg), lp_y=f64(n_seg), lq_y=f64(n_seg),
             lp_x=f64(n_seg), lq_x=f64(n_seg),
             status=torch.zeros(1, dtype=torch.int32, device=DEV))
    if per_row:
        t["lp0"] = f64(n_rows)
        t["lq"] = f64(n_rows)
    return t


@pytest.mark.parametrize("per_row", [False, True])
def test_no_alloc_matches_workspace_entry_point(per_row):
    w = make_workload(2, device=DEV, T=512, n_pf=12, seed=2024)
    assert w.n_rows <= 262144
    ref = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                  V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    ref.score()
    torch.cuda.synchronize()
    assert int(ref.t["status"].item()) == 0
    req = ~w.layout.is_root()
    want = {k: ref.t[k].cpu().numpy() for k in ("log_accept", "log_ratio", "lp0", "lq")}
    for call in range(2):                       # two calls in a row share the array
        t = _outputs(w.n_rows, w.layout.n_seg, per_row)
        out = ps.make_score_out(**t)
        ps.ps_score_subtree_noalloc(ref.batch, out)
        torch.cuda.synchronize()
        assert int(t["status"].item()) == 0, ps.dev_status_names(int(t["status"].item()))
        for k in ("log_accept", "log_ratio"):
            got = t[k].cpu().numpy()[req]
            assert np.all(np.abs(got - want[k][req]) <= H.LA_ATOL), (call, k)
        if per_row:
            for k in ("lp0", "lq"):
                got = t[k].cpu().numpy()
                assert np.all(np.abs(got - want[k]) <= H.TOK_RTOL * np.abs(want[k]) + 1e-300)


@pytest.mark.parametrize("supplied", ["lp0", "lq"])
def test_no_alloc_writes_the_one_per_row_array_supplied(supplied):
    # the other per-row array goes to the static array; the supplied one must
    # be written as ps_score_subtree writes it
    w = make_workload(2, device=DEV, T=256, n_pf=8, seed=2025)
    ref = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                  V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    ref.score()
    torch.cuda.synchronize()
    assert int(ref.t["status"].item()) == 0
    req = ~w.layout.is_root()
    want = ref.t[supplied].cpu().numpy()
    for call in range(2):
        t = _outputs(w.n_rows, w.layout.n_seg, per_row=False)
        t[supplied] = torch.full((w.n_rows,), float("nan"), dtype=torch.float64, device=DEV)
        ps.ps_score_subtree_noalloc(ref.batch, ps.make_score_out(**t))
        torch.cuda.synchronize()
        assert int(t["status"].item()) == 0, ps.dev_status_names(int(t["status"].item()))
        got = t[supplied].cpu().numpy()
        assert np.all(np.abs(got - want) <= H.TOK_RTOL * np.abs(want) + 1e-300), (call, supplied)
        la = t["log_accept"].cpu().numpy()[req]
        assert np.all(np.abs(la - ref.t["log_accept"].cpu().numpy()[req]) <= H.LA_ATOL)


def test_no_alloc_with_entropy_eps_classes_and_a_row_index():
    # rows read through a shuffled row index, the entropy of p0 and the
    # epsilon classes requested; 2,492 rows of 75 chunks each, so every
    # warp of the launch holds parts of rows that other warps finish, and the
    # split-row partials and counters live in the static array
    w0 = make_workload(2, device=DEV, T=320, n_pf=10, seed=2026)
    n = w0.n_rows
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(5)).to(DEV)
    pool = torch.empty_like(w0.logits)
    pool[perm] = w0.logits                  # row r of the batch sits at pool[perm[r]]
    ri = perm.to(torch.int64)
    assert n * ((w0.V * 2 + 4095) // 4096) > 4096
    f64 = lambda k: torch.empty(k, dtype=torch.float64, device=DEV)
    ref = ps.DeviceSubtree.create(layout=w0.layout, u=w0.u, logits=pool, tokens=w0.tokens,
                                  V=w0.V, alpha=w0.alpha, tau=w0.tau, max_steps=w0.max_steps,
                                  row_index=ri, entropy=True, eps=0.01)
    ref.score()
    torch.cuda.synchronize()
    assert int(ref.t["status"].item()) == 0
    req = ~w0.layout.is_root()
    n_seg = w0.layout.n_seg
    for call in range(2):
        t = _outputs(n, n_seg, per_row=False)
        t["entropy"] = f64(n)
        t["eps_class"] = torch.full((n_seg,), 9, dtype=torch.int8, device=DEV)
        ps.ps_score_subtree_noalloc(ref.batch, ps.make_score_out(**t))
        torch.cuda.synchronize()
        assert int(t["status"].item()) == 0, ps.dev_status_names(int(t["status"].item()))
        want_h = ref.t["entropy"].cpu().numpy()
        got_h = t["entropy"].cpu().numpy()
        assert np.all(np.abs(got_h - want_h) <= H.ENT_RTOL * np.abs(want_h) + H.ENT_ATOL), call
        for k in ("log_accept", "log_ratio"):
            got = t[k].cpu().numpy()[req]
            assert np.all(np.abs(got - ref.t[k].cpu().numpy()[req]) <= H.LA_ATOL), (call, k)
        assert torch.equal(t["eps_class"], ref.t["eps_class"]), call


def test_no_alloc_rejects_batches_beyond_its_row_limit():
    # a real, valid batch of 262145 rows (V = 8, 4 MB of logits): one root
    # segment with cut 0 and T = n_rows, so even a launch would stay in bounds
    n = 262145
    logits = torch.zeros((n, 8), dtype=torch.bfloat16, device=DEV)
    tokens = torch.zeros(n, dtype=torch.int32, device=DEV)
    b = ps.make_batch(V=8, T=n, alpha=4.0, tau=0.25,
                      chain_seg0=torch.tensor([0, 1], dtype=torch.int32, device=DEV),
                      seg_row0=torch.tensor([0, n], dtype=torch.int64, device=DEV),
                      seg_cut=torch.zeros(1, dtype=torch.int32, device=DEV),
                      seg_src=torch.full((1,), -1, dtype=torch.int32, device=DEV),
                      logits=logits, tokens=tokens)
    t = _outputs(0, 1, per_row=False)
    out = ps.make_score_out(**t)
    st = ps.ps_score_subtree_noalloc(b, out, check=False)
    assert st == 7          # PS_ERR_WORKSPACE, returned before anything is launched
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0
    assert torch.isnan(t["log_accept"]).all()     # untouched
    # nor with only one of the per-row outputs supplied: the other one would
    # need the static array
    for only in ("lp0", "lq"):
        t1 = _outputs(0, 1, per_row=False)
        t1[only] = torch.full((n,), float("nan"), dtype=torch.float64, device=DEV)
        assert ps.ps_score_subtree_noalloc(b, ps.make_score_out(**t1), check=False) == 7
        torch.cuda.synchronize()
        assert torch.isnan(t1[only]).all()
    # with both per-row outputs supplied there is no row limit
    t2 = _outputs(n, 1, per_row=True)
    out2 = ps.make_score_out(**t2)
    assert ps.ps_score_subtree_noalloc(b, out2, check=False) == 0
    torch.cuda.synchronize()
    assert int(t2["status"].item()) == 0
    assert torch.allclose(t2["lp0"], torch.full_like(t2["lp0"], -np.log(8.0)), rtol=1e-6)
