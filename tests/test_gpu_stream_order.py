"""Stream order with the caller's own kernels.

ps_assemble_subtree and ps_walk_subtree launch their kernels with
programmatic dependent launch, so those kernels may start while the previous
kernel in the stream is finishing.  The caller's inputs can come from such a
kernel: here a torch kernel rewrites the uniforms, the tree arrays or the
segment arrays immediately before the call, on the same stream, after a
kernel that filled them with wrong values.  The results must be those of a
run on inputs written long before (the walk and log A of the PreSTO round,
section 3.2 step (3) and eq. (6)).  The same holds for ps_score_walk_subtree,
whose suffix-sum + walk kernel reads the layout early.
"""

import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth import make_workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BIG = 1 << 24          # elements of the buffers the rewriting kernels cover


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _reference(w):
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    d.step()
    torch.cuda.synchronize()
    assert int(d.t["status"].item()) == 0 and int(d.t["wstatus"].item()) == 0
    return d


def _rewrite(dst_big: torch.Tensor, good_big: torch.Tensor, bad_big: torch.Tensor):
    """Two elementwise kernels over the whole buffer: wrong values, then the
    right ones (multiplying by 1 is exact for these dtypes)."""
    torch.mul(bad_big, 1, out=dst_big)
    torch.mul(good_big, 1, out=dst_big)


def test_uniforms_and_tree_written_by_a_kernel_just_before_the_walk():
    w = make_workload(2, device=DEV, T=64, n_pf=12, seed=91)
    ref = _reference(w)
    n_seg = int(ref.t["u"].shape[0])
    n_nodes = int(ref.t["acc"].shape[0])
    # u inside a large float64 buffer; bad uniforms reject... or accept, where
    # the right ones do the opposite
    ug = torch.zeros(BIG, dtype=torch.float64, device=DEV)
    ug[:n_seg] = ref.t["u"]
    ub = torch.ones(BIG, dtype=torch.float64, device=DEV)
    la = ref.t["log_accept"]
    ub[:n_seg] = torch.where(torch.rand(n_seg, dtype=torch.float64, device=DEV).log() <= la,
                             torch.ones_like(la), torch.full_like(la, 1e-300))
    u_buf = torch.empty(BIG, dtype=torch.float64, device=DEV)
    # the tree's rejection children inside a large int32 buffer; the bad copy
    # swaps them with the acceptance children
    rg = torch.zeros(BIG, dtype=torch.int32, device=DEV)
    rg[:n_nodes] = ref.t["rej"]
    rb = torch.zeros(BIG, dtype=torch.int32, device=DEV)
    rb[:n_nodes] = ref.t["acc"]
    r_buf = torch.empty(BIG, dtype=torch.int32, device=DEV)
    tree = ps.make_tree(chain_node0=ref.t["chain_node0"], chain_seg0=ref.t["chain_seg0"],
                        acc=ref.t["acc"], rej=r_buf[:n_nodes], req=ref.t["req"],
                        u=u_buf[:n_seg], max_steps=w.max_steps)
    n_ch = int(ref.t["k_delta"].shape[0])
    for it in range(20):
        out = {k: torch.full((n_ch,), -7, dtype=torch.int32, device=DEV)
               for k in ("state_seg", "end_node", "k_delta")}
        path = torch.full_like(ref.t["path"], -7)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        wout = ps.make_walk_out(state_seg=out["state_seg"], end_node=out["end_node"],
                                k_delta=out["k_delta"], status=status, path=path)
        if it % 2 == 0:
            _rewrite(r_buf, rg, rb)
            _rewrite(u_buf, ug, ub)        # the kernel right before the walk writes u
        else:
            _rewrite(u_buf, ug, ub)
            _rewrite(r_buf, rg, rb)        # ... or the tree
        ps.ps_walk_subtree(tree, la, wout)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, ps.dev_status_names(int(status.item()))
        for k in ("state_seg", "end_node", "k_delta"):
            assert torch.equal(out[k], ref.t[k]), (it, k)
        assert torch.equal(path, ref.t["path"]), it


def test_segments_written_by_a_kernel_just_before_the_suffix_sums():
    w = make_workload(2, device=DEV, T=64, n_pf=12, seed=92)
    ref = _reference(w)
    n_seg = int(ref.t["seg_cut"].shape[0])
    # seg_cut and seg_src side by side in one large int32 buffer; the bad copy
    # holds cuts and sources that fail the layout checks or change the sums
    good = torch.zeros(BIG, dtype=torch.int32, device=DEV)
    good[:n_seg] = ref.t["seg_cut"]
    good[n_seg:2 * n_seg] = ref.t["seg_src"]
    bad = torch.zeros(BIG, dtype=torch.int32, device=DEV)
    bad[:n_seg] = 1
    bad[n_seg:2 * n_seg] = torch.roll(ref.t["seg_src"], 1)
    buf = torch.empty(BIG, dtype=torch.int32, device=DEV)
    batch = ps.make_batch(V=w.V, T=w.layout.T, alpha=w.alpha, tau=w.tau,
                          chain_seg0=ref.t["chain_seg0"], seg_row0=ref.t["seg_row0"],
                          seg_cut=buf[:n_seg], seg_src=buf[n_seg:2 * n_seg],
                          logits=w.logits, tokens=w.tokens)
    for it in range(20):
        la = torch.full((n_seg,), 7.0, dtype=torch.float64, device=DEV)
        lr = torch.full((n_seg,), 7.0, dtype=torch.float64, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        sout = ps.make_score_out(log_accept=la, log_ratio=lr, status=status)
        _rewrite(buf, good, bad)
        ps.ps_assemble_subtree(batch, ref.t["lp0"], ref.t["lq"], sout)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, ps.dev_status_names(int(status.item()))
        req = torch.from_numpy(~w.layout.is_root()).to(DEV)
        assert torch.equal(la[req], ref.t["log_accept"][req]), it
        assert torch.equal(lr[req], ref.t["log_ratio"][req]), it
        assert bool(torch.isnan(la[~req]).all())


def test_inputs_written_by_a_kernel_just_before_the_one_call_round():
    # ps_score_walk_subtree launches its scoring kernel without early start, so
    # that kernel sees the caller's writes; the suffix-sum + walk kernel reads
    # the layout before waiting on the scoring kernel, which is only safe
    # because the caller's kernels finished before the scoring kernel began
    w = make_workload(2, device=DEV, T=64, n_pf=12, seed=93)
    ref = _reference(w)
    n_seg = int(ref.t["seg_cut"].shape[0])
    good = torch.zeros(BIG, dtype=torch.int32, device=DEV)
    good[:n_seg] = ref.t["seg_cut"]
    good[n_seg:2 * n_seg] = ref.t["seg_src"]
    bad = torch.zeros(BIG, dtype=torch.int32, device=DEV)
    bad[:n_seg] = 1
    bad[n_seg:2 * n_seg] = torch.roll(ref.t["seg_src"], 1)
    buf = torch.empty(BIG, dtype=torch.int32, device=DEV)
    ug = torch.zeros(BIG, dtype=torch.float64, device=DEV)
    ug[:n_seg] = ref.t["u"]
    ub = torch.full((BIG,), 1e-300, dtype=torch.float64, device=DEV)
    u_buf = torch.empty(BIG, dtype=torch.float64, device=DEV)
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    d.batch.seg_cut, d.batch.seg_src = buf[:n_seg].data_ptr(), buf[n_seg:2 * n_seg].data_ptr()
    d.tree.u = u_buf[:n_seg].data_ptr()
    d.batch._keep = d.batch._keep + (buf,)
    d.tree._keep = d.tree._keep + (u_buf,)
    req = torch.from_numpy(~w.layout.is_root()).to(DEV)
    for it in range(10):
        for k in ("status", "wstatus"):
            d.t[k].zero_()
        d.t["log_accept"].fill_(7.0)
        _rewrite(u_buf, ug, ub)
        _rewrite(buf, good, bad)                # the kernel right before the call
        d.step()
        torch.cuda.synchronize()
        st = int(d.t["status"].item()) | int(d.t["wstatus"].item())
        assert st == 0, ps.dev_status_names(st)
        assert torch.equal(d.t["log_accept"][req], ref.t["log_accept"][req]), it
        for k in ("state_seg", "end_node", "k_delta", "path"):
            assert torch.equal(d.t[k], ref.t[k]), (it, k)
