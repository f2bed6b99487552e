"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same bytes, and compare with the stated tolerances.

Tolerances (from the benchmark spec of the parity bar):
  per-token log-probabilities: |gpu - oracle| <= 1e-4 |oracle| (+1e-300 so
      that an exact 0 compares equal to -0);
  log A: |gpu - oracle| <= 1e-3 absolute;
  walk: path, end node, k_Delta and reached state identical, except after a
      decision with |log u - log A| < 1e-3, where the GPU walk must still be
      the walk its own log A values give;
  entropy of p0: |gpu - oracle| <= 1e-4 |oracle| + 2e-6 nats (float sums of
      up to 262144 terms, finalised in float64);
  epsilon classes: identical, except for decisions whose log A lies within
      1e-3 of log eps or log(1 - eps) (the log A tolerance).
"""

from __future__ import annotations

import numpy as np
import torch

import mh_prefetch_subtree_gb300 as ps
import oracle
from oracle.hostcopy import oracle_rows  # noqa: F401  (used by the tests too)

TOK_RTOL = 1e-4
TOK_ATOL = 1e-300
LA_ATOL = 1e-3
NEAR_TIE = 1e-3
ENT_RTOL = 1e-4
ENT_ATOL = 2e-6
EPS = 0.01


def run_gpu(w, per_row: bool = True, sums: bool = True, stream=None,
            entropy: bool = True) -> dict:
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                row_index=w.row_index, per_row=per_row, sums=sums,
                                entropy=entropy, eps=EPS)
    d.step(stream)
    torch.cuda.synchronize()
    out = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v)
           for k, v in d.t.items()
           if k in ("lp0", "lq", "lp_y", "lq_y", "lp_x", "lq_x", "log_ratio", "log_accept",
                    "status", "wstatus", "state_seg", "end_node", "k_delta", "path",
                    "entropy", "eps_class")
           and v is not None}
    out["status"] = int(out["status"][0])
    out["wstatus"] = int(out["wstatus"][0])
    return out


def run_oracle(w, threads: int | None = None, rows=None) -> dict:
    """The oracle on the workload; `rows` = (lp0, lq, entropy) per row when the
    caller already has the oracle's per-row values (e.g. of a row pool)."""
    lp0, lq, ent = oracle_rows(w, threads=threads) if rows is None else rows
    sums = oracle.suffix_sums(w.layout, lp0, lq)
    r, la = oracle.log_accept(sums, w.alpha)
    wk = oracle.walk(w.layout, la, w.u, w.max_steps)
    out = dict(lp0=lp0, lq=lq, entropy=ent, log_ratio=r, log_accept=la, walk=wk,
               eps_class=oracle.eps_class(la, EPS))
    out.update(sums)
    return out


def check_rows(g: dict, o: dict, rtol: float = TOK_RTOL) -> dict:
    stats = {}
    for k in ("lp0", "lq"):
        a, b = g[k], o[k]
        assert a.shape == b.shape
        assert np.array_equal(np.isnan(a), np.isnan(b)), f"{k}: NaN pattern differs"
        inf = np.isinf(b)          # a masked token: -inf on both sides
        assert np.array_equal(a[inf], b[inf]), f"{k}: infinite values differ"
        m = ~np.isnan(b) & ~inf
        err = np.abs(a[m] - b[m])
        bound = rtol * np.abs(b[m]) + TOK_ATOL
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, (f"{k}: {bad.size} rows off; worst rel "
                               f"{np.max(err / (np.abs(b[m]) + 1e-300)):.3e}")
        rel = err / np.maximum(np.abs(b[m]), 1e-300)
        stats[f"{k}_max_rel"] = float(rel.max()) if rel.size else 0.0
    if g.get("entropy") is not None:
        a, b = g["entropy"], o["entropy"]
        assert np.array_equal(np.isnan(a), np.isnan(b)), "entropy: NaN pattern differs"
        m = ~np.isnan(b)
        err = np.abs(a[m] - b[m])
        bad = np.nonzero(err > ENT_RTOL * np.abs(b[m]) + ENT_ATOL)[0]
        assert bad.size == 0, f"entropy: {bad.size} rows off; worst |diff| {err.max():.3e}"
        stats["entropy_max_abs"] = float(err.max()) if err.size else 0.0
    return stats


def check_log_accept(w, g: dict, o: dict, atol: float = LA_ATOL) -> dict:
    req = ~w.layout.is_root()
    stats = {}
    for k in ("log_accept", "log_ratio"):
        a, b = g[k][req], o[k][req]
        assert np.array_equal(np.isnan(a), np.isnan(b)), f"{k}: NaN pattern differs"
        m = ~np.isnan(b)
        err = np.abs(a[m] - b[m])
        assert (err <= atol).all(), f"{k}: max |diff| {err.max():.3e}"
        stats[f"{k}_max_abs"] = float(err.max()) if err.size else 0.0
    for k in ("lp_y", "lq_y", "lp_x", "lq_x"):
        if k in g:
            a, b = g[k][req], o[k][req]
            err = np.abs(a - b)
            stats[f"{k}_max_abs"] = float(np.nanmax(err)) if err.size else 0.0
    if g.get("eps_class") is not None:
        gc, oc = g["eps_class"], o["eps_class"]
        assert np.all(gc[~req] == -1)
        la = o["log_accept"]
        near = ((np.abs(la - np.log(EPS)) < LA_ATOL) | (np.abs(la - np.log1p(-EPS)) < LA_ATOL))
        diff = (gc != oc) & req
        assert not np.any(diff & ~near), "epsilon classes differ away from the thresholds"
        stats["eps_class_near_threshold"] = int(np.sum(diff))
    return stats


def check_walk(w, g: dict, o: dict) -> dict:
    """Walk parity with the near-tie rule."""
    lay = w.layout
    mine = oracle.walk(lay, g["log_accept"], w.u, w.max_steps)   # GPU log A, oracle walk
    stride = w.max_steps + 1
    near = 0
    for c in range(lay.n_chains):
        gp = g["path"][c * stride:(c + 1) * stride]
        k = int(g["k_delta"][c])
        gpath = list(gp[:k + 1])
        assert all(x == -1 for x in gp[k + 1:])
        # the GPU walk is the walk its own log A values give
        assert gpath == mine["path"][c]
        assert int(g["state_seg"][c]) == int(mine["state_seg"][c])
        assert int(g["end_node"][c]) == int(mine["end_node"][c])
        opath = o["walk"]["path"][c]
        if gpath != opath:
            i = next(j for j in range(min(len(gpath), len(opath))) if gpath[j] != opath[j])
            s = int(lay.req[gpath[i - 1]])
            gap = abs(np.log(w.u[s]) - o["log_accept"][s])
            assert gap < NEAR_TIE, f"chain {c}: walks differ at a decision {gap:.3e} from a tie"
            near += 1
        else:
            assert int(g["k_delta"][c]) == int(o["walk"]["k_delta"][c])
            assert int(g["state_seg"][c]) == int(o["walk"]["state_seg"][c])
    return dict(walk_near_ties=near, k_delta_mean=float(np.mean(g["k_delta"])))


def full_parity(w, threads: int | None = None, rows=None) -> dict:
    """The round computed twice, with the entropy of p0 and without it (the
    two kinds of scoring kernel: without entropy, large batches take tail
    blocks), each compared with one oracle run.  The stats of the run without
    entropy carry the suffix "_no_entropy"."""
    o = None
    stats = {}
    for entropy in (True, False):
        g = run_gpu(w, entropy=entropy)
        assert g["status"] == 0, ps.dev_status_names(g["status"])
        assert g["wstatus"] == 0, ps.dev_status_names(g["wstatus"])
        if o is None:
            o = run_oracle(w, threads=threads, rows=rows)
        s = {}
        s.update(check_rows(g, o))
        s.update(check_log_accept(w, g, o))
        s.update(check_walk(w, g, o))
        stats.update(s if entropy else {k + "_no_entropy": v for k, v in s.items()})
    stats["eps_certain"] = oracle.eps_certain_fraction(o["log_accept"][~w.layout.is_root()])
    return stats
