"""Calls from several host threads on their own streams (the header's
thread-safety statement): each thread's results equal those of the same
batch scored alone, bit for bit (the path is deterministic)."""

import threading

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth import make_workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
KEYS = ("lp0", "lq", "log_accept", "state_seg", "k_delta", "entropy")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _subtree(w):
    return ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                   V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                   entropy=True, eps=0.01)


def _results(d):
    return {k: d.t[k].cpu().numpy().copy() for k in KEYS}


def test_concurrent_host_threads_on_own_streams():
    ws = [make_workload(2, device=DEV, T=256, n_pf=8, seed=300 + i) for i in range(4)]
    alone = []
    for w in ws:
        d = _subtree(w)
        d.step()
        torch.cuda.synchronize()
        alone.append(_results(d))
    subs = [_subtree(w) for w in ws]
    errors = []

    def run(i):
        try:
            s = torch.cuda.Stream(device=DEV)
            for _ in range(5):
                subs[i].step(s)
            s.synchronize()
        except Exception as e:          # reported below
            errors.append(e)

    th = [threading.Thread(target=run, args=(i,)) for i in range(len(ws))]
    for t in th:
        t.start()
    for t in th:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for d, ref in zip(subs, alone):
        assert int(d.t["status"].item()) == 0 and int(d.t["wstatus"].item()) == 0
        got = _results(d)
        for k in KEYS:
            assert np.array_equal(got[k], ref[k], equal_nan=True), k
