"""GPU parity of the round carry-over (section 3.2 step (3)) and of scoring a
round whose current state is carried from the previous round instead of
re-scored."""

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
import oracle
from synth import make_workload
from synth.trees import assemble_layout, bfs_tree
from synth.workload import Workload, draw_tokens, gen_logits
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def _device(w, entropy=True, **kw):
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                row_index=w.row_index, entropy=entropy, eps=0.01, **kw)
    d.step()
    torch.cuda.synchronize()
    assert int(d.t["status"].item()) == 0 and int(d.t["wstatus"].item()) == 0
    return d


@pytest.mark.parametrize("cfg,kw", [(1, {}), (2, dict(T=256, n_pf=8, seed=5)),
                                    (2, dict(T=128, n_pf=6, seed=6, n_chains=5))])
def test_carry_matches_oracle(cfg, kw):
    w = make_workload(cfg, device=DEV, **kw)
    d = _device(w)
    lay = w.layout
    rng = np.random.default_rng(7)
    prev = {k: rng.normal(size=(lay.n_chains, lay.T)) for k in ("lp0", "lq", "entropy")}
    prev_t = {k: torch.from_numpy(v).to(DEV) for k, v in prev.items()}
    g = d.carry(prev_t)
    torch.cuda.synchronize()
    assert int(g["status"].item()) == 0
    o_rows = H.oracle_rows(w)
    state = d.t["state_seg"].cpu().numpy()
    o = oracle.carry_state(lay, state, {"lp0": o_rows[0], "lq": o_rows[1], "entropy": o_rows[2]},
                           prev)
    for k in ("lp0", "lq"):
        a, b = g[k].cpu().numpy(), o[k]
        assert np.all(np.abs(a - b) <= H.TOK_RTOL * np.abs(b) + 1e-300), k
    a, b = g["entropy"].cpu().numpy(), o["entropy"]
    assert np.all(np.abs(a - b) <= H.ENT_RTOL * np.abs(b) + H.ENT_ATOL)
    np.testing.assert_allclose(g["loglik"].cpu().numpy(), o["loglik"], rtol=1e-4, atol=1e-7)
    np.testing.assert_allclose(g["confidence"].cpu().numpy(), o["confidence"], rtol=1e-4,
                               atol=1e-7)


def _first_round(T, V, seed):
    rng = np.random.default_rng(seed)
    tree = bfs_tree(rng, T, 8)
    tree.finalize_root_cut(0)                  # the root has rows for every position
    lay = assemble_layout([tree])
    x = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), lay.n_rows, V, "bf16",
                   seed=seed + 1, device=DEV)
    tok = draw_tokens(x, 0.25, seed=seed + 2)
    return Workload(name="first MH round", layout=lay, V=V, dtype="bf16", alpha=4.0, tau=0.25,
                    logits=x, tokens=tok, u=1.0 - rng.random(lay.n_seg), max_steps=100)


def test_second_round_with_a_carried_current_state():
    T, V = 384, 151936
    for seed in (11, 12, 13):
        w1 = _first_round(T, V, seed)
        d1 = _device(w1, entropy=False)
        carried = d1.carry()
        torch.cuda.synchronize()
        assert int(carried["status"].item()) == 0
        # the second MH round: a fresh subtree rooted at the reached state
        rng = np.random.default_rng(seed + 100)
        tree2 = bfs_tree(rng, T, 6)
        u2 = 1.0 - rng.random(len(tree2.seg_cut))
        tree2.finalize_root_cut(T)                 # (A) carried: no root rows
        lay_a = assemble_layout([tree2])
        xr = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), lay_a.n_rows, V, "bf16",
                        seed=seed + 3, device=DEV)
        tr = draw_tokens(xr, 0.25, seed=seed + 4)
        wa = Workload(name="carried", layout=lay_a, V=V, dtype="bf16", alpha=4.0, tau=0.25,
                      logits=xr, tokens=tr, u=u2, max_steps=100)
        da = _device(wa, entropy=False, root_lp0=carried["lp0"], root_lq=carried["lq"])
        # (B) the same round with the reached state's rows scored again
        st = oracle.materialize(w1.layout, 0)
        s_star = int(d1.t["state_seg"].item())
        node = next(i for i, x in enumerate(st.state_seg) if x == s_star and st.rows[i] is not None)
        rows1 = torch.from_numpy(st.rows[node][1:]).to(DEV)
        tree2.finalize_root_cut(0)
        lay_b = assemble_layout([tree2])
        wb = Workload(name="rows", layout=lay_b, V=V, dtype="bf16", alpha=4.0, tau=0.25,
                      logits=torch.cat([w1.logits[rows1], xr]),
                      tokens=torch.cat([w1.tokens[rows1], tr]), u=u2, max_steps=100)
        db = _device(wb, entropy=False)
        la_a = da.t["log_accept"].cpu().numpy()[1:]
        la_b = db.t["log_accept"].cpu().numpy()[1:]
        assert np.max(np.abs(la_a - la_b)) <= 1e-4
        # and both against the oracle with the oracle's own carried values
        o1 = H.run_oracle(w1)
        oc = oracle.carry_state(w1.layout, np.array([s_star]), {"lp0": o1["lp0"], "lq": o1["lq"]},
                                {})
        o_rows = H.oracle_rows(wa)
        sums = oracle.suffix_sums(lay_a, o_rows[0], o_rows[1], root_lp0=oc["lp0"],
                                  root_lq=oc["lq"])
        _, la_o = oracle.log_accept(sums, 4.0)
        assert np.max(np.abs(la_a - la_o[1:])) <= H.LA_ATOL
        assert int(da.t["k_delta"].item()) == int(db.t["k_delta"].item())
