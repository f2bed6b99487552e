"""Diagnostics on the GPU.  Failure detection without a fault: a bounded
device wait that nothing completes ends with PS_DEV_TIMEOUT, and the context
stays usable.  The plain-read probe that the bench times reads every word of
its buffer once."""

import time

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth import make_workload
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
PS_DEV_TIMEOUT = 0x20


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ps.ps_selftest_wait_timeout(50_000_000, status)         # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == PS_DEV_TIMEOUT
    assert 0.045 <= dt < 5.0, dt
    # the context is still usable: a scoring pass right after it is correct
    w = make_workload(1, device=DEV)
    s = H.full_parity(w)
    assert s["lp0_max_rel"] <= H.TOK_RTOL
    # and a second timeout on another stream reports again
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream(device=DEV)
    ps.ps_selftest_wait_timeout(2_000_000, st2, side)
    torch.cuda.synchronize()
    assert int(st2.item()) == PS_DEV_TIMEOUT


def test_read_probe_reads_every_word_once():
    # the plain-read diagnostic folds every 32-bit word of the buffer with XOR:
    # equal to numpy's fold over the same bytes, for a buffer whose length is
    # not a multiple of the probe's stride
    import numpy as np
    g = torch.Generator(device="cuda:0")
    g.manual_seed(7)
    n = (1 << 20) * 37 + 12
    x = torch.randint(-2**31, 2**31 - 1, (n,), dtype=torch.int32, device="cuda:0", generator=g)
    sink = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    ps.ps_selftest_read(x, sink)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(x.cpu().numpy().view(np.uint32))
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want)
