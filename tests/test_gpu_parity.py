"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every case compares element by element on the same seeded bytes: per-token
log-probabilities within 1e-4 relative, log A within 1e-3 absolute, and the
walk exactly (near-ties excepted, see tests/gpu_harness.py).
"""

import math

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
import oracle
from synth import make_workload
from synth.trees import assemble_layout, bfs_tree
from synth.workload import (SWEEP5, Workload, draw_tokens, gen_logits, make_pool,
                             sweep_pool_rows, workload_config5)
from tests import gpu_harness as H
from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _report(name, stats):
    print(f"\n[{name}] " + " ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                                  for k, v in stats.items()))


# ---- the five configurations ----------------------------------------------

def test_config1_tiny_full():
    w = make_workload(1, device=DEV)
    _report("config1", H.full_parity(w))


def test_config2_full():
    w = make_workload(2, device=DEV)
    _report("config2", H.full_parity(w))


def test_config3_full():
    w = make_workload(3, device=DEV)
    s = H.full_parity(w)
    s["suffix_tokens"] = w.info["suffix_tokens"]
    _report("config3", s)
    assert 90_000 <= w.info["suffix_tokens"] <= 110_000


def test_config4_full():
    # the peaked-logits configuration is calibrated (sigma_b = 4.5) so that 67-95%
    # of the decisions are epsilon-certain (A <= 0.01 or A >= 0.99)
    w = make_workload(4, device=DEV)
    s = H.full_parity(w)
    _report("config4", s)
    assert 0.67 <= s["eps_certain"] <= 0.95


@pytest.fixture(scope="module")
def sweep_pool():
    """The row pool of configuration 5, as the bench builds it (at least 16 GB
    of distinct rows and 128 x the L2 size), and the oracle's per-row values of
    every pool row at each sweep temperature (tokens are drawn per (row, tau),
    so a scored row's values depend only on its pool row and tau)."""
    taus = [1.0 / a for a in SWEEP5["alpha"]]
    n_pool = sweep_pool_rows(SWEEP5["V"], 2, torch.cuda.get_device_properties(DEV).L2_cache_size)
    pool, ptok = make_pool(n_pool, SWEEP5["V"], "bf16", SWEEP5["logits"][1], taus,
                           seed=10091, device=DEV)
    lg = bf16_bits(pool)
    vals = {}
    for t in taus:
        vals[float(t)] = oracle.row_logprobs(lg, "bf16", SWEEP5["V"], ptok[float(t)].cpu().numpy(),
                                             t, entropy=True)
    return pool, ptok, vals


@pytest.mark.parametrize("T", SWEEP5["T"])
@pytest.mark.parametrize("n_pf", SWEEP5["n_pf"])
@pytest.mark.parametrize("alpha", SWEEP5["alpha"])
def test_config5_sweep_point(sweep_pool, n_pf, T, alpha):
    # 256 independent chains; rows read through a shuffled row index into a pool
    # of distinct rows (> L2); every scored row is compared
    pool, ptok, vals = sweep_pool
    w = workload_config5(pool, ptok, n_pf, T, alpha, n_chains=256)
    ri = w.row_index.cpu().numpy()
    lp0, lq, ent = vals[float(w.tau)]
    s = H.full_parity(w, rows=(lp0[ri], lq[ri], ent[ri]))
    _report(f"config5 Npf={n_pf} T={T} a={alpha}", s)


# ---- shapes, temperatures, edge cases ---------------------------------------

def _small(V, dtype, T=12, n_pf=5, tau=0.25, alpha=4.0, n_chains=2, seed=0, kind="boosted",
           sigma=3.0, ld=None, max_steps=100):
    rng = np.random.default_rng(seed)
    trees = [bfs_tree(rng, T, n_pf) for _ in range(n_chains)]
    lay = assemble_layout(trees)
    u = 1.0 - rng.random(lay.n_seg)
    params = dict(sigma=sigma, margin_mean=4.0)
    ldv = V if ld is None else ld
    x = gen_logits(kind, params, lay.n_rows, V, dtype, seed=seed + 1, device=DEV)
    if ldv != V:
        big = torch.full((lay.n_rows, ldv), float("nan"), dtype=x.dtype, device=DEV)
        big[:, :V] = x
        x = big
    tok = draw_tokens(x, tau, seed=seed + 2, V=V)
    return Workload(name="small", layout=lay, V=V, dtype=dtype, alpha=alpha, tau=tau, logits=x,
                    tokens=tok, u=u, max_steps=max_steps)


@pytest.mark.parametrize("V,dtype,ld", [
    (1, "f32", 4), (2, "bf16", 8), (7, "bf16", 8), (1000, "bf16", 1008), (1000, "f32", 1000),
    (2048, "bf16", None), (2056, "bf16", None), (4097, "f32", 4100), (151936, "bf16", None),
    (262144, "bf16", None), (65536 + 24, "bf16", 65536 + 32), (151936, "f32", None),
    (151937, "bf16", 151944)])
def test_vocab_shapes_and_padding(V, dtype, ld):
    # NaN padding beyond V must be ignored (it is patched to -inf in shared memory);
    # a one-token vocabulary cannot hold a boosted token, so it uses plain rows
    w = _small(V, dtype, ld=ld, seed=V, kind="normal" if V == 1 else "boosted")
    _report(f"V={V} {dtype} ld={ld}", H.full_parity(w))


@pytest.mark.parametrize("tau,alpha", [(1.0, 1.0), (0.5, 2.0), (0.25, 4.0), (0.125, 8.0),
                                       (0.3, 4.0), (2.0, 0.5), (0.7, 1.5)])
def test_temperatures(tau, alpha):
    w = _small(151936, "bf16", T=20, n_pf=6, tau=tau, alpha=alpha, seed=int(tau * 1000))
    _report(f"tau={tau}", H.full_parity(w))


def test_many_rows_few_warps_and_split_rows():
    # one long row per chain, many chains: rows split across many warps
    w = _small(262144, "bf16", T=2, n_pf=1, n_chains=3, seed=5)
    _report("split", H.full_parity(w))
    # more rows than warps, ragged last chunk of every row
    w = _small(5000, "bf16", T=64, n_pf=16, n_chains=40, seed=6)
    _report("many rows", H.full_parity(w))


def test_dominant_token_keeps_relative_accuracy():
    # margin 30 over all others: lq ~ -1e-50 must still match to 1e-4 relative
    for V, dtype in ((151936, "bf16"), (1024, "f32")):
        w = _small(V, dtype, T=6, n_pf=2, n_chains=1, seed=9)
        x = torch.zeros_like(w.logits)
        rows = torch.arange(w.n_rows, device=DEV)
        x[rows, w.tokens.long()] = 30.0
        w.logits = x
        g = H.run_gpu(w)
        o = H.run_oracle(w)
        s = H.check_rows(g, o)
        _report(f"dominant {dtype}", s)
        assert (o["lq"] < 0).all() and (o["lq"] > -1e-40).all()


def test_entropy_edge_cases():
    # uniform rows (H = log V), one-token rows (H = 0), a peaked row, masked
    # entries and a masked token: entropy and log-probabilities against the oracle
    V = 151936
    w = _small(V, "bf16", T=8, n_pf=3, n_chains=1, seed=21)
    x = w.logits.clone()
    x[0] = 0.5                                   # uniform
    x[1] = float("-inf")
    x[1, 5] = 2.0                                # a single finite logit
    w.tokens[1] = 5
    x[2] = 0.0
    x[2, 9] = 30.0                               # peaked
    x[3, 2000:] = float("-inf")                  # masked tail
    w.logits = x
    g = H.run_gpu(w)
    o = H.run_oracle(w)
    s = H.check_rows(g, o)
    _report("entropy edges", s)
    assert abs(g["entropy"][0] - np.log(V)) < 1e-4 and g["entropy"][1] == 0.0


@pytest.mark.parametrize("V,dtype", [(151936, "bf16"), (262144, "bf16"), (4100, "f32")])
def test_entropy_of_peaked_rows_whose_token_is_not_the_peak(V, dtype):
    # one logit far above the rest, placed anywhere in the row (often in a late
    # chunk), and the token elsewhere: the entropy is small and the sum of
    # 2^y y cancels against S1 log2 S1, so this checks that the dominant term is
    # accumulated close to the reference
    w = _small(V, dtype, T=12, n_pf=4, n_chains=2, seed=23, kind="normal")
    n = w.n_rows
    rng = np.random.default_rng(24)
    x = w.logits.clone()
    peak = torch.from_numpy(rng.integers(0, V, n)).to(DEV)
    margin = torch.from_numpy(rng.choice([3.0, 6.0, 10.0, 15.0, 25.0, 40.0], n)).to(DEV)
    rows = torch.arange(n, device=DEV)
    x[rows, peak] = (x[:, :V].float().max(dim=1).values + margin.float()).to(x.dtype)
    tok = torch.from_numpy(rng.integers(0, V, n).astype(np.int32)).to(DEV)
    tok = torch.where(tok.long() == peak, (tok + 1) % V, tok)
    w.logits, w.tokens = x, tok
    g = H.run_gpu(w)
    o = H.run_oracle(w)
    s = H.check_rows(g, o)
    _report(f"peaked off-token {V} {dtype}", s)
    assert np.median(o["entropy"]) < 0.5


def test_masked_vocabulary():
    w = _small(151936, "bf16", T=10, n_pf=4, n_chains=2, seed=11)
    x = w.logits.clone()
    x[:, 1000:] = float("-inf")             # only the first 1000 ids allowed
    w.logits = x
    w.tokens = draw_tokens(x, w.tau, seed=12)
    _report("masked", H.full_parity(w))


def test_masked_vocabulary_with_the_masked_hint():
    # PS_FLAG_MASKED_LOGITS changes only how the entropy variant sums: results
    # match the oracle as without it
    w = _small(151936, "bf16", T=10, n_pf=4, n_chains=2, seed=15)
    x = w.logits.clone()
    x[:, 2000:] = float("-inf")
    x[0, :] = float("-inf")
    x[0, 7] = 1.0                                # one finite logit
    w.logits = x
    w.tokens = draw_tokens(x, w.tau, seed=16)
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                entropy=True, eps=H.EPS, flags=ps.PS_FLAG_MASKED_LOGITS)
    d.step()
    torch.cuda.synchronize()
    assert int(d.t["status"].item()) == 0
    g = {k: d.t[k].cpu().numpy() for k in ("lp0", "lq", "entropy")}
    _report("masked hint", H.check_rows(g, H.run_oracle(w)))


def test_status_bits_and_nan_outputs():
    w = _small(4096, "bf16", T=8, n_pf=3, n_chains=1, seed=13)
    tok = w.tokens.clone()
    tok[0] = 4096                            # out of range
    x = w.logits.clone()
    x[1, 17] = float("nan")                  # NaN logit
    w.tokens, w.logits = tok, x
    g = H.run_gpu(w)
    assert g["status"] & 0x01 and g["status"] & 0x02
    assert np.isnan(g["lp0"][0]) and np.isnan(g["lp0"][1])
    assert np.isfinite(g["lp0"][2:]).all()


def test_infeasible_request_is_flagged():
    w = _small(1024, "f32", T=10, n_pf=4, n_chains=1, seed=14)
    lay = w.layout
    # make request 2 claim a from-state whose cut is below its own (Condition 1)
    bad = None
    for s in range(1, lay.n_seg):
        for t in range(1, lay.n_seg):
            if t != s and lay.seg_cut[t] < lay.seg_cut[s]:
                bad = (s, t)
                break
        if bad:
            break
    assert bad is not None
    lay.seg_src = lay.seg_src.copy()
    lay.seg_src[bad[0]] = bad[1]
    g = H.run_gpu(w)
    assert g["status"] & 0x04
    assert np.isnan(g["log_accept"][bad[0]])


def test_bad_row_index_is_flagged():
    pool = gen_logits("normal", dict(sigma=1.0), 16, 2048, "bf16", seed=3, device=DEV)
    rng = np.random.default_rng(15)
    lay = assemble_layout([bfs_tree(rng, 6, 2)])
    ri = torch.from_numpy(rng.integers(0, 16, lay.n_rows)).to(DEV)
    ri[0] = 99
    tok = torch.zeros(lay.n_rows, dtype=torch.int32, device=DEV)
    w = Workload(name="ri", layout=lay, V=2048, dtype="bf16", alpha=4.0, tau=0.25, logits=pool,
                 tokens=tok, u=np.ones(lay.n_seg), max_steps=10, row_index=ri)
    g = H.run_gpu(w)
    assert g["status"] & 0x40 and np.isnan(g["lp0"][0]) and np.isfinite(g["lp0"][1:]).all()


def test_bit_reproducible():
    w = make_workload(2, device=DEV, T=256, n_pf=8, seed=99)
    a = H.run_gpu(w)
    b = H.run_gpu(w)
    for k in ("lp0", "lq", "log_accept", "k_delta", "path"):
        assert np.array_equal(a[k], b[k], equal_nan=True)


def test_alpha_tau_one_full_size():
    # alpha = tau = 1 accepts everything (r = 0) at the full configuration-2 size
    w = make_workload(2, device=DEV, alpha=1.0, tau=1.0)
    g = H.run_gpu(w)
    req = ~w.layout.is_root()
    assert np.max(np.abs(g["log_ratio"][req])) <= 1e-3
    assert (g["k_delta"] >= 1).all()


def test_copied_suffix_full_size():
    # proposals that copy their from-state's rows give r = 0 (eq. (6))
    w = make_workload(2, device=DEV, n_pf=8, seed=123)
    lay = w.layout
    st = oracle.materialize(lay, 0)
    x, tok = w.logits, w.tokens
    for v in range(lay.n_nodes):
        s = int(lay.req[v])
        if s < 0:
            continue
        cs = int(lay.seg_cut[s])
        src_rows = torch.from_numpy(st.rows[v][cs + 1:]).to(DEV)
        dst = torch.arange(int(lay.seg_row0[s]), int(lay.seg_row0[s + 1]), device=DEV)
        x[dst] = x[src_rows]
        tok[dst] = tok[src_rows]
    g = H.run_gpu(w)
    req = ~lay.is_root()
    assert np.max(np.abs(g["log_ratio"][req])) <= 1e-3
    assert (g["log_accept"][req] > -1e-3).all()


# ---- the walk on its own ------------------------------------------------------

def _walk_only(lay, logA, u, max_steps):
    d = {k: torch.as_tensor(np.ascontiguousarray(getattr(lay, k), dtype=np.int32)).to(DEV)
         for k in ("chain_node0", "chain_seg0", "acc", "rej", "req")}
    tree = ps.make_tree(u=torch.as_tensor(u).to(DEV), max_steps=max_steps, **d)
    nc = lay.n_chains
    out = {k: torch.empty(nc, dtype=torch.int32, device=DEV)
           for k in ("state_seg", "end_node", "k_delta")}
    out["status"] = torch.zeros(1, dtype=torch.int32, device=DEV)
    out["path"] = torch.empty(nc * (max_steps + 1), dtype=torch.int32, device=DEV)
    wo = ps.make_walk_out(**out)
    la = torch.as_tensor(logA).to(DEV)
    ps.ps_walk_subtree(tree, la, wo)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_walk_brute_force_patterns():
    rng = np.random.default_rng(41)
    import itertools
    checked = 0
    while checked < 20:
        lay = assemble_layout([bfs_tree(rng, int(rng.integers(2, 9)), int(rng.integers(1, 7)))])
        nreq = lay.n_seg - 1
        if nreq < 1:
            continue
        logA = np.concatenate([[np.nan], np.log(rng.uniform(0.05, 0.95, nreq))])
        A = np.exp(logA)
        pats = list(itertools.product((0, 1), repeat=nreq))
        # one chain per pattern, all in one launch
        from synth.trees import assemble_layout as asm
        lays = asm(lay.trees * len(pats))
        u = np.ones(lays.n_seg)
        for p_i, bits in enumerate(pats):
            for s in range(1, lay.n_seg):
                u[p_i * lay.n_seg + s] = A[s] / 2 if bits[s - 1] else (1 + A[s]) / 2
        la = np.tile(logA, len(pats))
        g = _walk_only(lays, la, u, 100)
        o = oracle.walk(lays, la, u, 100)
        assert g["status"][0] == 0
        assert np.array_equal(g["k_delta"], o["k_delta"])
        assert np.array_equal(g["state_seg"], o["state_seg"])
        assert np.array_equal(g["end_node"], o["end_node"])
        for c in range(lays.n_chains):
            assert list(g["path"][c * 101:c * 101 + o["k_delta"][c] + 1]) == o["path"][c]
        checked += 1


def test_walk_decisions_at_tiny_acceptance_probabilities():
    # one request per chain, log A and u chosen around the walk's shortcuts:
    # below log A = -80 every u >= 1e-30 rejects without an exponential; a
    # smaller u, or a u within 1e-5 of A, is settled by the float64 one
    from synth.trees import ChainTree
    cases = [(-85.0, 1e-30), (-85.0, 0.5), (-85.0, math.exp(-86.0)), (-85.0, math.exp(-84.0)),
             (-80.0, 1e-30), (-80.0, math.exp(-80.0) * (1 - 1e-9)),
             (-79.9, math.exp(-79.9) * (1 - 1e-6)), (-79.9, math.exp(-79.9) * (1 + 1e-6)),
             (-200.0, 1e-300), (-700.0, 1e-300), (-700.0, 1e-305), (-745.0, 1e-320),
             (-math.inf, 5e-324),
             (-1e-12, 1.0), (-3.0, math.exp(-3.0) * (1 - 1e-7))]
    trees = []
    for _ in cases:
        t = ChainTree.new(16)
        t.expand(0, 5)
        t.finalize_root_cut()
        trees.append(t)
    lay = assemble_layout(trees)
    la = np.full(lay.n_seg, np.nan)
    u = np.ones(lay.n_seg)
    for c, (a, x) in enumerate(cases):
        la[2 * c + 1], u[2 * c + 1] = a, x
    g = _walk_only(lay, la, u, 10)
    o = oracle.walk(lay, la, u, 10)
    assert g["status"][0] == 0
    want = np.array([1 if x <= math.exp(a) else 0 for a, x in cases])
    assert list(want) == [0, 0, 1, 0, 0, 1, 1, 0, 1, 0, 1, 0, 0, 0, 1]
    assert np.array_equal(o["k_delta"], np.ones(len(cases)))
    accepted = g["state_seg"] == np.arange(len(cases)) * 2 + 1
    assert np.array_equal(accepted.astype(int), want)
    assert np.array_equal(g["state_seg"], o["state_seg"])
    assert np.array_equal(g["end_node"], o["end_node"])


def test_walk_max_steps_deferred_and_cycle():
    rng = np.random.default_rng(42)
    lay = assemble_layout([bfs_tree(rng, 10, 6) for _ in range(50)])
    la = np.zeros(lay.n_seg)
    u = np.full(lay.n_seg, 0.5)
    for m in (0, 1, 3, 100):
        g = _walk_only(lay, la, u, m)
        o = oracle.walk(lay, la, u, m)
        assert np.array_equal(g["k_delta"], o["k_delta"]) and g["status"][0] == 0
    # a cycle: point the first acceptance child back to the root
    bad = assemble_layout([bfs_tree(np.random.default_rng(1), 10, 3)])
    bad.acc = bad.acc.copy()
    bad.req = bad.req.copy()
    a = int(bad.acc[0])
    bad.req[a] = bad.req[0]       # the child asks the same request, then loops
    bad.acc[a] = 0
    g = _walk_only(bad, np.zeros(bad.n_seg), np.full(bad.n_seg, 0.5), 1000)
    assert g["status"][0] & 0x08
