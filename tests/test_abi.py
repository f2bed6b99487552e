"""The C ABI on the CPU: the library loads, exports every function include/ps.h
declares, and its host-side checks and validator behave (no GPU calls)."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import mh_prefetch_subtree_gb300 as ps
from synth.trees import DEFERRED, assemble_layout, bfs_tree, example5_tree

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from mh_prefetch_subtree_gb300.build import build
    build()


def declared_functions():
    with open(os.path.join(ROOT, "include", "ps.h")) as fh:
        src = fh.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ps_[a-z_]+)\s*\(", src)))


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert len(names) >= 8
    out = subprocess.check_output(["nm", "-D", "--defined-only", ps.LIB_PATH], text=True)
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    L = ps.lib()
    for n in names:
        assert hasattr(L, n)


def test_struct_sizes_match_the_header_layout():
    # int32 x6, int64 x3, double x3, 9 pointers
    assert ctypes.sizeof(ps.PsSubtreeBatch) == 6 * 4 + 3 * 8 + 3 * 8 + 9 * 8
    assert ctypes.sizeof(ps.PsCarryIo) == 13 * 8
    assert ctypes.sizeof(ps.PsScoreOut) == 11 * 8
    assert ctypes.sizeof(ps.PsTree) == 4 * 4 + 6 * 8
    assert ctypes.sizeof(ps.PsWalkOut) == 5 * 8


def test_status_strings():
    assert ps.ps_status_string(0) == "ok"
    assert "Condition 1" in ps.ps_status_string(2)
    assert ps.ps_status_string(99) == "unknown status"
    assert "sm_103a" in ps.ps_version()


def _host(layout, V=64, tokens=None):
    b = ps.make_batch(V=V, T=layout.T, alpha=4.0, tau=0.25,
                      chain_seg0=np.ascontiguousarray(layout.chain_seg0),
                      seg_row0=np.ascontiguousarray(layout.seg_row0),
                      seg_cut=np.ascontiguousarray(layout.seg_cut),
                      seg_src=np.ascontiguousarray(layout.seg_src),
                      tokens=tokens, n_rows=layout.n_rows, n_logit_rows=layout.n_rows)
    t = ps.make_tree(chain_node0=np.ascontiguousarray(layout.chain_node0),
                     chain_seg0=np.ascontiguousarray(layout.chain_seg0),
                     acc=np.ascontiguousarray(layout.acc), rej=np.ascontiguousarray(layout.rej),
                     req=np.ascontiguousarray(layout.req), u=np.ones(layout.n_seg), max_steps=10)
    return b, t


def test_validator_accepts_generated_batches():
    rng = np.random.default_rng(1)
    for _ in range(50):
        T = int(rng.integers(1, 40))
        lay = assemble_layout([bfs_tree(rng, T, int(rng.integers(0, 12)))
                               for _ in range(int(rng.integers(1, 5)))])
        tok = rng.integers(0, 64, lay.n_rows).astype(np.int32)
        b, t = _host(lay, tokens=tok)
        st, msg = ps.ps_validate_subtree(b, t)
        assert st == 0, msg


def test_validator_rejects_infeasible_and_bad_layouts():
    lay = assemble_layout([example5_tree(20, 9, 4)])
    # Condition 1: request z (cut 4, from y at cut 9) made to claim cut 12 > 9
    cut = lay.seg_cut.copy()
    cut[2] = 12
    rows = lay.seg_row0.copy()
    rows[3] = rows[2] + (20 - 12)
    lay2 = assemble_layout([example5_tree(20, 9, 4)])
    lay2.seg_cut, lay2.seg_row0 = cut, rows
    b, t = _host(lay2)
    b.n_rows = int(rows[-1])
    st, msg = ps.ps_validate_subtree(b, None)
    assert st == 2, msg
    # wrong src for the tree (z claims to come from the root)
    src = lay.seg_src.copy()
    src[2] = 0
    lay3 = assemble_layout([example5_tree(20, 9, 4)])
    lay3.seg_src = src
    b, t = _host(lay3)
    st, msg = ps.ps_validate_subtree(b, t)
    assert st == 3 and "seg_src" in msg
    # segment size that is not T - cut
    lay4 = assemble_layout([example5_tree(20, 9, 4)])
    lay4.seg_row0 = lay4.seg_row0.copy()
    lay4.seg_row0[1] += 1
    b, t = _host(lay4)
    st, msg = ps.ps_validate_subtree(b, None)
    assert st == 1 and "rows" in msg
    # token out of range
    b, t = _host(lay, tokens=np.full(lay.n_rows, 64, np.int32))
    st, msg = ps.ps_validate_subtree(b, None)
    assert st == 1 and "token" in msg


def test_validator_rejects_bad_trees():
    lay = assemble_layout([example5_tree(20, 9, 4)])
    for mutate in ("two_parents", "cycle", "reuse_request", "bad_code"):
        acc, rej, req = lay.acc.copy(), lay.rej.copy(), lay.req.copy()
        if mutate == "two_parents":
            rej[1] = 2
        elif mutate == "cycle":
            acc[3] = 1
        elif mutate == "reuse_request":
            req[2] = 1
            acc[2], rej[2] = 3, 4
        elif mutate == "bad_code":
            req[4] = -7
        t = ps.make_tree(chain_node0=lay.chain_node0, chain_seg0=lay.chain_seg0, acc=acc,
                         rej=rej, req=req, u=np.ones(lay.n_seg), max_steps=5)
        st, msg = ps.ps_validate_subtree(None, t)
        assert st == 3, (mutate, msg)


def test_deferred_nodes_validate():
    rng = np.random.default_rng(3)
    seen = 0
    for _ in range(40):
        lay = assemble_layout([bfs_tree(rng, 8, 6)])
        seen += int((lay.req == DEFERRED).sum())
        b, t = _host(lay)
        assert ps.ps_validate_subtree(b, t)[0] == 0
    assert seen > 0


def test_host_argument_checks_need_no_gpu():
    import torch
    lay = assemble_layout([example5_tree(8, 5, 2)])
    b, _ = _host(lay)
    ws = torch.zeros(16, dtype=torch.uint8)
    out = ps.PsScoreOut()
    # missing outputs / bad header are rejected before any CUDA call
    assert ps.ps_score_subtree(b, out, ws, check=False, stream=0) == 1
    b.V = 0
    assert ps.ps_score_subtree(b, out, ws, check=False, stream=0) == 1
    b.V = 64
    b.tau = -1.0
    assert ps.ps_score_subtree(b, out, ws, check=False, stream=0) == 1
    b.tau = 0.25
    b.dtype = 7
    assert ps.ps_score_subtree(b, out, ws, check=False, stream=0) == 4
    assert ps.ps_score_workspace_bytes(b) > 0


def test_multi_temperature_host_checks_need_no_gpu():
    import torch
    lay = assemble_layout([example5_tree(8, 5, 2)])
    b, _ = _host(lay)
    logits = torch.zeros(lay.n_rows, 64, dtype=torch.bfloat16)
    toks = torch.zeros(lay.n_rows, dtype=torch.int32)
    b.logits = logits.data_ptr()
    b.tokens = toks.data_ptr()
    lp0 = torch.zeros(lay.n_rows, dtype=torch.float64)
    status = torch.zeros(1, dtype=torch.int32)
    ws = torch.zeros(16, dtype=torch.uint8)

    def call(taus):
        lq = torch.zeros(len(taus), lay.n_rows, dtype=torch.float64)
        return ps.ps_score_rows_multi(b, taus, lp0, lq, status, ws, check=False, stream=0)

    # 1/tau outside {1, 2, 4, 8}, or more than four temperatures: unsupported
    assert call([0.25, 0.3]) == 4
    assert call([1.0, 0.5, 0.25, 0.125, 1.0]) == 4
    assert call([]) == 4
    # a temperature that is not a positive finite number: invalid argument
    assert call([0.25, -0.5]) == 1
    assert call([float("nan")]) == 1
    # supported temperatures pass the checks and stop at the workspace size
    assert call([0.25, 0.5, 1.0]) == 7


def test_wait_selftest_host_checks_need_no_gpu():
    import torch
    st = torch.zeros(1, dtype=torch.int32)
    # limits outside 1 us .. 2 s are rejected before any CUDA call
    assert ps.ps_selftest_wait_timeout(10, st, stream=0, check=False) == 1
    assert ps.ps_selftest_wait_timeout(3_000_000_000, st, stream=0, check=False) == 1
    # a host pointer is not device memory
    assert ps.ps_selftest_wait_timeout(1_000_000, st, stream=0, check=False) == 1


def test_row_size_limit_needs_no_gpu():
    import torch
    lay = assemble_layout([example5_tree(8, 5, 2)])
    b, _ = _host(lay)
    logits = torch.zeros(lay.n_rows, 64, dtype=torch.bfloat16)
    toks = torch.zeros(lay.n_rows, dtype=torch.int32)
    b.logits, b.tokens = logits.data_ptr(), toks.data_ptr()
    lp0 = torch.zeros(lay.n_rows, dtype=torch.float64)
    lq = torch.zeros(lay.n_rows, dtype=torch.float64)
    st = torch.zeros(1, dtype=torch.int32)
    ws = torch.zeros(16, dtype=torch.uint8)

    def call():
        return ps.ps_score_rows(b, lp0, lq, st, ws, stream=0, check=False)

    assert call() == 7                       # header accepted; stops at the workspace
    b.V = b.ld = 1 << 29                     # bf16 rows of exactly 2^30 bytes: allowed
    assert call() == 7
    b.V = b.ld = (1 << 29) + 8               # above 2^30 bytes
    assert call() == 1
    b.dtype, b.V, b.ld = 1, (1 << 28) + 4, (1 << 28) + 4
    assert call() == 1


def test_batch_flags_need_no_gpu():
    import torch
    lay = assemble_layout([example5_tree(8, 5, 2)])
    b, _ = _host(lay)
    logits = torch.zeros(lay.n_rows, 64, dtype=torch.bfloat16)
    toks = torch.zeros(lay.n_rows, dtype=torch.int32)
    b.logits, b.tokens = logits.data_ptr(), toks.data_ptr()
    lp0 = torch.zeros(lay.n_rows, dtype=torch.float64)
    lq = torch.zeros(lay.n_rows, dtype=torch.float64)
    st = torch.zeros(1, dtype=torch.int32)
    ws = torch.zeros(16, dtype=torch.uint8)
    b.flags = ps.PS_FLAG_MASKED_LOGITS          # a known hint: passes to the workspace check
    assert ps.ps_score_rows(b, lp0, lq, st, ws, stream=0, check=False) == 7
    b.flags = 0x2                               # an unknown bit
    assert ps.ps_score_rows(b, lp0, lq, st, ws, stream=0, check=False) == 1


def test_read_probe_host_checks_need_no_gpu():
    import torch
    sink = torch.zeros(1, dtype=torch.int32)
    data = torch.zeros(64, dtype=torch.uint8)
    # a size that is not a multiple of 16 bytes, and a misaligned start
    assert ps.ps_selftest_read(data[:40], sink, stream=0, check=False) == 1
    assert ps.ps_selftest_read(data[4:36], sink, stream=0, check=False) == 1
    # a host pointer is not device memory
    assert ps.ps_selftest_read(data[:32], sink, stream=0, check=False) == 1
