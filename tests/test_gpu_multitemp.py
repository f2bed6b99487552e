"""GPU parity of multi-temperature row scoring (ps_score_rows_multi).

MultiTryMH as the PreSTO pages run it (section 5.1; Appendix D.4, Table 6(a))
draws each candidate suffix at a temperature from {0.25, 0.5, 1.0}; one pass
over a row gives log q_tau of its token at all of them.  Each temperature is
compared with the oracle's plain definition at that tau, row by row, within
the per-token tolerance (1e-4 relative); entropy within its own tolerance.
"""

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
import oracle
from synth.trees import assemble_layout, bfs_tree
from synth.workload import draw_tokens, gen_logits
from tests import gpu_harness as H
from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TABLE6_TAUS = [0.25, 0.5, 1.0]


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _rows(V, dtype, taus, T=12, n_pf=5, n_chains=2, seed=0, ld=None, kind="boosted"):
    """A subtree batch whose rows' tokens are drawn at a temperature picked per
    row from `taus` (the candidates of one MultiTryMH transition)."""
    rng = np.random.default_rng(seed)
    lay = assemble_layout([bfs_tree(rng, T, n_pf) for _ in range(n_chains)])
    ldv = V if ld is None else ld
    x = gen_logits(kind, dict(sigma=3.0, margin_mean=4.0), lay.n_rows, V, dtype,
                   seed=seed + 1, device=DEV)
    if ldv != V:
        big = torch.full((lay.n_rows, ldv), float("nan"), dtype=x.dtype, device=DEV)
        big[:, :V] = x
        x = big
    pick = rng.integers(0, len(taus), lay.n_rows)
    tok = torch.empty(lay.n_rows, dtype=torch.int32, device=DEV)
    for k, t in enumerate(taus):
        tk = draw_tokens(x, t, seed=seed + 2 + k, V=V)
        sel = torch.from_numpy(np.nonzero(pick == k)[0]).to(DEV)
        tok[sel] = tk[sel]
    d = ps.DeviceSubtree.create(layout=lay, u=1.0 - rng.random(lay.n_seg), logits=x, tokens=tok,
                                V=V, alpha=4.0, tau=0.25, max_steps=10, entropy=True)
    return d, x, tok


def _run_multi(d, taus, entropy=True):
    n = d.batch.n_rows
    lp0 = torch.full((n,), float("nan"), dtype=torch.float64, device=DEV)
    lq = torch.full((len(taus), n), float("nan"), dtype=torch.float64, device=DEV)
    ent = torch.full((n,), float("nan"), dtype=torch.float64, device=DEV) if entropy else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ps.ps_score_rows_multi(d.batch, taus, lp0, lq, status, d.workspace, entropy=ent)
    torch.cuda.synchronize()
    return (lp0.cpu().numpy(), lq.cpu().numpy(),
            None if ent is None else ent.cpu().numpy(), int(status.item()))


def _oracle(x, dtype, V, tok, tau):
    lg = bf16_bits(x) if dtype == "bf16" else x.cpu().numpy()
    return oracle.row_logprobs(lg, dtype, V, tok.cpu().numpy(), tau, entropy=True)


def _check(a, b, what):
    g = {"lp0": a[0], "lq": a[1], "entropy": a[2]}
    o = {"lp0": b[0], "lq": b[1], "entropy": b[2]}
    try:
        return H.check_rows(g, o)
    except AssertionError as e:
        raise AssertionError(f"{what}: {e}") from None


@pytest.mark.parametrize("V,dtype,ld", [
    (151936, "bf16", None), (262144, "bf16", None), (1000, "f32", 1000), (7, "bf16", 8),
    (4097, "f32", 4100), (2056, "bf16", None)])
@pytest.mark.parametrize("taus", [TABLE6_TAUS, [0.125, 0.25, 0.5, 1.0], [0.5], [1.0, 0.125]])
def test_multi_temperature_matches_oracle(V, dtype, ld, taus):
    d, x, tok = _rows(V, dtype, taus, seed=V % 97 + len(taus), ld=ld)
    lp0, lq, ent, status = _run_multi(d, taus)
    assert status == 0, ps.dev_status_names(status)
    for k, t in enumerate(taus):
        o = _oracle(x, dtype, V, tok, t)
        _check((lp0, lq[k], ent), o, f"tau={t}")


def test_multi_temperature_split_rows_and_many_rows():
    # long rows split across warps (merged through the workspace partials) and
    # many short rows with a ragged last chunk
    for V, T, n_pf, chains in ((262144, 2, 1, 3), (5000, 64, 16, 40)):
        d, x, tok = _rows(V, "bf16", TABLE6_TAUS, T=T, n_pf=n_pf, n_chains=chains, seed=V)
        lp0, lq, ent, status = _run_multi(d, TABLE6_TAUS)
        assert status == 0
        for k, t in enumerate(TABLE6_TAUS):
            _check((lp0, lq[k], ent), _oracle(x, "bf16", V, tok, t), f"V={V} tau={t}")


def test_multi_agrees_with_single_temperature_calls():
    taus = [0.125, 0.25, 0.5, 1.0]
    d, x, tok = _rows(151936, "bf16", taus, T=16, n_pf=6, seed=3)
    lp0, lq, ent, status = _run_multi(d, taus)
    assert status == 0
    n = d.batch.n_rows
    for k, t in enumerate(taus):
        d.batch.tau = t
        s_lp0 = torch.empty(n, dtype=torch.float64, device=DEV)
        s_lq = torch.empty(n, dtype=torch.float64, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        ps.ps_score_rows(d.batch, s_lp0, s_lq, st, d.workspace)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        np.testing.assert_allclose(lq[k], s_lq.cpu().numpy(), rtol=H.TOK_RTOL, atol=0)
        np.testing.assert_allclose(lp0, s_lp0.cpu().numpy(), rtol=H.TOK_RTOL, atol=0)
    # tau = 1 is p0 itself: the same float sum, so the same value
    assert np.array_equal(lq[taus.index(1.0)], lp0)


def test_multi_without_entropy_and_dominant_token():
    # margin 30: log q at tau = 1/8 is about -1e-100 and must keep its
    # relative accuracy
    taus = [0.125, 0.25, 1.0]
    for V, dtype in ((151936, "bf16"), (1024, "f32")):
        d, x, tok = _rows(V, dtype, taus, T=6, n_pf=2, n_chains=1, seed=9)
        y = torch.zeros_like(x)
        y[torch.arange(x.shape[0], device=DEV), tok.long()] = 30.0
        x.copy_(y)
        lp0, lq, _, status = _run_multi(d, taus, entropy=False)
        assert status == 0
        for k, t in enumerate(taus):
            o = _oracle(x, dtype, V, tok, t)
            _check((lp0, lq[k], None), (o[0], o[1], None), f"dominant tau={t}")
            assert (o[1] < 0).all()


def test_multi_status_bits_and_nan_rows():
    d, x, tok = _rows(4096, "bf16", TABLE6_TAUS, T=8, n_pf=3, n_chains=1, seed=13)
    tok[0] = 4096                       # out of range
    x[1, 17] = float("nan")             # NaN logit
    lp0, lq, ent, status = _run_multi(d, TABLE6_TAUS)
    assert status & 0x01 and status & 0x02
    for r in (0, 1):
        assert np.isnan(lp0[r]) and np.isnan(lq[:, r]).all() and np.isnan(ent[r])
    assert np.isfinite(lp0[2:]).all() and np.isfinite(lq[:, 2:]).all()


def test_multi_rejects_unsupported_temperatures():
    d, _, _ = _rows(1000, "f32", [1.0], T=4, n_pf=1, n_chains=1, seed=2)
    n = d.batch.n_rows
    lp0 = torch.empty(n, dtype=torch.float64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for taus in ([0.3], [0.25, 0.7], [1.0] * 5):
        lq = torch.empty(len(taus), n, dtype=torch.float64, device=DEV)
        assert ps.ps_score_rows_multi(d.batch, taus, lp0, lq, st, d.workspace,
                                      check=False) == ps.PS_ERR_UNSUPPORTED


def test_multi_temperature_through_a_row_index():
    # rows read through a shuffled row index into a pool (the sweep's layout):
    # every temperature against the oracle on the pool row each scored row reads
    V = 151936
    rng = np.random.default_rng(31)
    n_pool = 600
    pool = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), n_pool, V, "bf16", seed=32,
                      device=DEV)
    lay = assemble_layout([bfs_tree(rng, 40, 6) for _ in range(8)])
    ri = torch.from_numpy(rng.integers(0, n_pool, lay.n_rows).astype(np.int64)).to(DEV)
    tok = torch.from_numpy(rng.integers(0, V, lay.n_rows).astype(np.int32)).to(DEV)
    d = ps.DeviceSubtree.create(layout=lay, u=1.0 - rng.random(lay.n_seg), logits=pool,
                                tokens=tok, V=V, alpha=4.0, tau=0.25, max_steps=10,
                                row_index=ri, entropy=True)
    lp0, lq, ent, status = _run_multi(d, TABLE6_TAUS)
    assert status == 0
    lg = bf16_bits(pool)
    for k, t in enumerate(TABLE6_TAUS):
        o = oracle.row_logprobs(lg, "bf16", V, tok.cpu().numpy(), t,
                                row_index=ri.cpu().numpy(), entropy=True)
        _check((lp0, lq[k], ent), o, f"row_index tau={t}")


@pytest.mark.parametrize("V,dtype", [(151936, "bf16"), (4097, "f32")])
def test_multi_temperature_on_masked_rows_with_and_without_the_hint(V, dtype):
    d, x, tok = _rows(V, dtype, TABLE6_TAUS, T=10, n_pf=4, n_chains=2, seed=41,
                      ld=4100 if dtype == "f32" else None)
    x[:, 700:V] = float("-inf")                       # a masked vocabulary
    tok.copy_(tok % 700)
    for flags in (0, ps.PS_FLAG_MASKED_LOGITS):
        d.batch.flags = flags
        lp0, lq, ent, status = _run_multi(d, TABLE6_TAUS)
        assert status == 0
        for k, t in enumerate(TABLE6_TAUS):
            _check((lp0, lq[k], ent), _oracle(x, dtype, V, tok, t), f"flags={flags} tau={t}")


def test_multi_temperature_with_tail_blocks_at_full_size():
    # configuration 4 (45,820 rows of 128 chunks) is large enough for tail
    # blocks in the variant without entropy; every row that reaches into the
    # last 1/16 of the chunks (the tail blocks) and 2,000 of the others are
    # compared with the oracle at each temperature
    from synth import make_workload
    w = make_workload(4, device=DEV)
    warps = torch.cuda.get_device_properties(0).multi_processor_count * 16
    assert w.n_rows * 128 >= 2048 * warps, "the batch is too small to have tail blocks"
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    lp0, lq, ent, status = _run_multi(d, TABLE6_TAUS, entropy=False)
    assert status == 0, ps.dev_status_names(status)
    assert ent is None
    n = w.n_rows
    tail0 = n - n // 16 - 1
    rng = np.random.default_rng(5)
    sel = np.unique(np.concatenate([np.arange(tail0, n), rng.choice(tail0, 2000, replace=False)]))
    idx = torch.from_numpy(sel).to(DEV)
    xs, ts = w.logits[idx], w.tokens[idx]
    for k, t in enumerate(TABLE6_TAUS):
        o = _oracle(xs, "bf16", w.V, ts, t)
        _check((lp0[sel], lq[k][sel], None), (o[0], o[1], None), f"tau={t}")
    del d, w
    torch.cuda.empty_cache()
