"""The round captured in a CUDA graph and replayed.

A caller that runs many small rounds (few rows per batch) is bound by launch
overhead; capturing ps_score_walk_subtree once and replaying the graph removes
the host-side cost of each call.  The replayed round must give exactly the
outputs of the eager call, and must read its inputs afresh at every replay
(here: new acceptance uniforms written into the same buffer between replays,
which change the walk of PreSTO section 3.2 step (3)).
"""

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth import make_workload
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
OUT = ("lp0", "lq", "lp_y", "lq_y", "lp_x", "lq_x", "log_ratio", "log_accept", "entropy",
       "eps_class", "state_seg", "end_node", "k_delta", "path", "status", "wstatus")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _snapshot(d):
    return {k: d.t[k].clone() for k in OUT if d.t.get(k) is not None}


def _poison(d):
    for k in OUT:
        t = d.t.get(k)
        if t is None:
            continue
        if k in ("status", "wstatus"):
            t.zero_()
        elif t.dtype.is_floating_point:
            t.fill_(float("nan"))
        else:
            t.fill_(-7)


def _same(a, b):
    for k in a:
        x, y = a[k].cpu().numpy(), b[k].cpu().numpy()
        assert np.array_equal(x, y, equal_nan=np.issubdtype(x.dtype, np.floating)), k


@pytest.mark.parametrize("case", ["config1", "config2_small"])
def test_captured_round_replays_the_eager_round(case):
    if case == "config1":
        w = make_workload(1, device=DEV)
    else:
        w = make_workload(2, device=DEV, T=64, n_pf=8, seed=51)
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                entropy=True, eps=H.EPS)
    s = torch.cuda.Stream(device=DEV)
    with torch.cuda.stream(s):
        d.step(s)                           # first call on the device, outside capture
    torch.cuda.synchronize()
    eager = _snapshot(d)
    assert int(eager["status"].item()) == 0 and int(eager["wstatus"].item()) == 0

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        d.step(s)
    for _ in range(2):
        _poison(d)
        g.replay()
        torch.cuda.synchronize()
        _same(eager, _snapshot(d))

    # new uniforms in the same buffer: the replay must walk with them
    rng = np.random.default_rng(52)
    u2 = 1.0 - rng.random(w.layout.n_seg)
    d.t["u"].copy_(torch.from_numpy(u2))
    _poison(d)
    g.replay()
    torch.cuda.synchronize()
    replayed = _snapshot(d)
    _poison(d)
    with torch.cuda.stream(s):
        d.step(s)
    torch.cuda.synchronize()
    _same(_snapshot(d), replayed)
