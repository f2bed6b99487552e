"""Benchmark: scoring one prefetched subtree batch (and walking it) on GB300.

One step = the whole hot path over one subtree batch already resident in HBM,
in one call (ps_score_walk_subtree): per-token log p0 / log q_tau of every
row, suffix sums and log A per request, and the walk of every chain.

Default workload: the long-context batch, the largest of the five
configurations that a single GPU holds: Qwen3-like vocabulary V = 151936
bf16, T = 3072, N_pf = 64 requests in a unary-heavy subtree (spine of depth
30), alpha = 4, tau = 0.25; 98,469 rows, 95,486 scored suffix tokens and
29.9 GB of logits, far larger than the 129 MB L2, so no flush is needed
between steps.

metric  scored suffix tokens per second (sum over requests of T - c_i,
        whole job over all ranks); logits GB/s and the HBM roofline of the
        scoring kernel are reported alongside.  The line also carries the
        scoring kernel's other variants, the end-to-end rate from host
        buffers, the CPU oracle on the same batch, and the 36-point throughput
        sweep (256 chains per point, rows read through a shuffled row index
        into a pool of distinct rows sized far above the L2).
Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun every rank scores its own batch (independent problems, weak
scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "scored suffix tokens/sec and logits GB/s vs GB300 HBM peak per subtree batch"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0            # the roofline the target is stated against
FALLBACK_HBM_GBS = 6800.0           # used only when MEASURED_PEAKS.json is absent
# DRAM bytes (read + write) per launch of the scoring kernel on the default
# workload, from one ncu capture of this kernel code (identified by its hash).
NCU_TRAFFIC = {"source_sha1": "5cb170908f66cd1a695bef1deab314f034cf2fef",
               "bytes_per_launch": 29925604608 + 7847680, "config": 3}
GENERAL_TAU = 0.3                   # a temperature whose 1/tau is not 1, 2, 4 or 8


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (a no-op without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: int, world_size: int, steps: int, max_ms: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return units_per_rank_step * world_size * steps / (max_ms / 1e3)


def rank_seed(config: int, rank: int):
    """Seed of each rank's batch: rank 0 uses the configuration's own seed, the
    others independent seeds, so the ranks score different batches."""
    return None if rank == 0 else 10086 + config + 7919 * rank


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha1() -> str:
    """Hash of the scoring kernel's code (its two source files with comments,
    blank lines and trailing blanks removed): the ncu traffic below is
    reported only while the code it was captured from is unchanged."""
    import re
    h = hashlib.sha1()
    for name in ("ps_score_rows.cu", "ps_internal.cuh"):
        with open(os.path.join(ROOT, "mh_prefetch_subtree_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        lines = [ln.rstrip() for ln in src.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        inside = [r for t, r in self.rows if self.t0 is not None and self.t0 <= t <= self.t1]
        use = inside if inside else [r for _, r in self.rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        mx = [num(r[2]) for r in use if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_region": len(inside),
                "power_w_max": max((num(r[3]) or 0.0) for r in use)}


def build_workload(config: int, dev, rank: int, n_pf=None):
    from synth import make_workload
    kw = {}
    if n_pf is not None:
        kw["n_pf"] = n_pf
    seed = rank_seed(config, rank)
    if seed is not None:
        kw["seed"] = seed
    return make_workload(config, device=dev, **kw)


def host_memory_available() -> int | None:
    """MemAvailable of /proc/meminfo in bytes, or None where it cannot be read."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def cpu_baseline(w, max_seconds: float = 30.0) -> tuple[dict, dict]:
    """The oracle, as it stands, on the same batch: per-row log-probabilities
    (the step computes no entropy, so neither does this), the suffix sums over
    explicit states, log A and the walk, on all host cores; and the per-row
    part on one core over a sample of rows, extrapolated to the batch.
    Returns the oracle's results (for the parity check) and the record."""
    import oracle
    from oracle.hostcopy import oracle_rows     # block-wise host copies for the oracle
    threads = oracle.default_threads()
    lay = w.layout
    units = lay.suffix_tokens()
    t0 = time.time()
    lp0, lq, _ent = oracle_rows(w, threads=threads, entropy=False)
    t1 = time.time()
    sums = oracle.suffix_sums(lay, lp0, lq)
    _, la = oracle.log_accept(sums, w.alpha)
    wk = oracle.walk(lay, la, w.u, w.max_steps)
    t2 = time.time()
    ref = dict(lp0=lp0, lq=lq, log_accept=la, walk=wk)
    dt = t2 - t0
    # one core: time growing row samples until one takes over max_seconds / 6
    n1, tr1 = 64, 0.0
    while True:
        s0 = time.time()
        oracle_rows(w, threads=1, entropy=False, n_rows=n1)
        tr1 = time.time() - s0
        if tr1 > max_seconds / 6 or n1 >= w.n_rows:
            break
        n1 = min(w.n_rows, n1 * 4)
    one_core_s = tr1 * w.n_rows / n1 + (t2 - t1)
    return ref, {"value": units / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu": cpu_model(), "nproc": os.cpu_count(),
            "sample": f"the whole batch ({w.n_rows} rows, {units} suffix tokens), "
                      f"{dt:.1f} s wall on {threads} threads",
            "one_core": {"value": units / one_core_s, "unit": UNIT, "cores": 1,
                         "sample": f"per-row part timed on {n1} rows ({tr1:.1f} s) and "
                                   f"scaled to {w.n_rows}; sums and walk as measured"}}


def parity_vs_oracle(w, d, ref) -> dict:
    """The timed batch's GPU results against the oracle's on the same bytes:
    worst per-token relative errors, worst log A error, and walks compared
    chain by chain (a walk may differ only after a decision whose log u lies
    within 1e-3 of log A, a near-tie)."""
    lay = w.layout
    req = ~lay.is_root()
    out = {}
    for k in ("lp0", "lq"):
        g, o = d.t[k].cpu().numpy(), ref[k]
        m = np.isfinite(o)
        out[f"{k}_max_rel"] = float(np.max(np.abs(g[m] - o[m]) / np.maximum(np.abs(o[m]), 1e-300)))
    la_g = d.t["log_accept"].cpu().numpy()
    out["log_accept_max_abs"] = float(np.max(np.abs(la_g[req] - ref["log_accept"][req])))
    wk = ref["walk"]
    state, kd = d.t["state_seg"].cpu().numpy(), d.t["k_delta"].cpu().numpy()
    differ = int(np.sum((state != wk["state_seg"]) | (kd != wk["k_delta"])))
    ties = 0
    for c in range(lay.n_chains):
        for v in wk["path"][c][:-1]:
            s = int(lay.req[v])
            if s >= 0 and abs(np.log(w.u[s]) - ref["log_accept"][s]) < 1e-3:
                ties += 1
    import oracle
    out.update({"walks_differing": differ, "near_ties_on_oracle_paths": ties,
                "eps_certain": oracle.eps_certain_fraction(ref["log_accept"][req]),
                "tolerances": "per token 1e-4 relative, log A 1e-3 absolute",
                "checked": f"all {lay.n_rows} rows and {int(req.sum())} requests of the batch"})
    return out


def reference_sample_tree(tree, row_budget: int):
    """A sample of one chain's subtree with at most about row_budget rows.

    Normally the root's rows and the first requests in order, request rows up
    to min(2,500, row_budget - root rows), at least one request.  When the
    root and the first request alone exceed row_budget, the sample is one
    request of the tree proposed from the root: the longest suffix whose two
    segments (root rows c+1..T and the request's) fit the budget, else the
    shortest one, with the root's cut raised to that request's cut.
    """
    from synth.trees import ChainTree
    T = tree.T
    root_rows = T - tree.seg_cut[0]
    cuts = tree.seg_cut[1:]
    if not cuts or root_rows + T - cuts[0] <= row_budget:
        budget = min(2500, row_budget - root_rows)
        keep, req_rows = 1, 0
        while keep < len(tree.seg_cut) and (
                keep == 1 or req_rows + T - tree.seg_cut[keep] <= budget):
            req_rows += T - tree.seg_cut[keep]
            keep += 1
        tree.seg_cut = tree.seg_cut[:keep]
        tree.seg_src = tree.seg_src[:keep]
        tree.req = [r if r < keep else -1 for r in tree.req]
        return tree
    fit = [c for c in cuts if 2 * (T - c) <= row_budget]
    c = min(fit) if fit else max(cuts)
    t = ChainTree.new(T)
    t.expand(0, c)
    t.finalize_root_cut()
    return t


def reference_arm(args, ws, rank):
    """--impl reference: the CPU oracle timed as the step, on bounded samples."""
    if rank != 0:
        return 0
    import oracle
    from synth import make_workload
    from synth.trees import assemble_layout
    w = make_workload(args.config, device="cpu") if args.config == 1 else None
    tokens_per_row = None               # of the full batch, when w is a sample of it
    if w is None:
        # a bounded sample of the same batch, sized so that the whole run stays
        # near 90 s at about 7,000 oracle rows/s on 16 cores (and a step at
        # most the root's rows + 2,500 request rows); tokens are credited at
        # the full batch's suffix tokens per row
        from synth.workload import CONFIGS, _trees_for, draw_tokens, gen_logits, Workload
        cfg = dict(CONFIGS[args.config])
        rng = np.random.default_rng(10086 + args.config)
        tree = _trees_for(cfg, rng)[0]
        full = assemble_layout([tree])
        tokens_per_row = full.suffix_tokens() / full.n_rows
        root_cut0 = tree.seg_cut[0]
        tree = reference_sample_tree(tree, 90 * 7000 // max(1, args.steps + args.warmup))
        lay = assemble_layout([tree])
        x = gen_logits(cfg["logits"][0], cfg["logits"][1], lay.n_rows, cfg["V"], cfg["dtype"],
                       seed=1, device="cpu")
        tok = draw_tokens(x, cfg["tau"], seed=2)
        w = Workload(name=cfg["name"], layout=lay, V=cfg["V"], dtype=cfg["dtype"],
                     alpha=cfg["alpha"], tau=cfg["tau"], logits=x, tokens=tok,
                     u=1.0 - rng.random(lay.n_seg), max_steps=cfg["max_steps"])
    from oracle.hostcopy import logits_np
    lg, dt = logits_np(w.logits)
    toks = w.tokens.numpy()
    threads = oracle.default_threads()

    def step():
        res = oracle.score_subtree(lg, dt, w.V, toks, w.layout, w.alpha, w.tau, threads=threads)
        oracle.walk(w.layout, res["log_accept"], w.u, w.max_steps)

    for _ in range(args.warmup):
        step()
    t0 = time.time()
    for _ in range(args.steps):
        step()
    el = time.time() - t0
    # The oracle's time is proportional to the rows it scores.  A sample keeps
    # all of the root's rows, so it holds more root rows per request row than
    # the batch; each sampled row is credited with the batch's suffix tokens
    # per row, so that the rate is the one the whole batch would give.
    if tokens_per_row is None:
        units_per_step = w.layout.suffix_tokens()
        how = f"the whole batch ({w.n_rows} rows) per step"
    else:
        units_per_step = w.n_rows * tokens_per_row
        which = ("the root's and its first requests'" if w.layout.seg_cut[0] == root_cut0
                 else "one request proposed from the root and the root's rows it reads")
        how = (f"{w.n_rows} rows of the batch per step ({which}); "
               f"tokens = rows x the batch's {tokens_per_row:.4f} suffix tokens per row")
    v = units_per_step * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample_rows": w.n_rows,
                       "sample_suffix_tokens": w.layout.suffix_tokens(),
                       "credited_tokens_per_step": units_per_step},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": how},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def sweep_leg(ps, dev, stream, steps: int, warmup: int, per_point: bool = False,
              max_points: int | None = None) -> dict:
    """The throughput sweep: at each of the 36 points (N_pf x T x alpha, tau =
    1/alpha) 256 independent chains, their rows read through a shuffled row
    index into a pool of distinct logits rows of at least 16 GB and 128 x the
    L2 size, so that the reads come from DRAM.  Each point's step (score,
    assemble, walk) and its scoring kernel alone are timed with CUDA events;
    the aggregate is the sum of tokens (and logits bytes) over the sum of
    times.  per_point prints one JSON line per point as well."""
    from synth.workload import SWEEP5, make_pool, sweep_pool_rows, workload_config5
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_pool = sweep_pool_rows(SWEEP5["V"], 2, l2)
    taus = [1.0 / a for a in SWEEP5["alpha"]]
    pool, ptok = make_pool(n_pool, SWEEP5["V"], "bf16", SWEEP5["logits"][1], taus, seed=10091,
                           device=dev)
    tot = dict(tokens=0, rows=0, ms=0.0, k1_ms=0.0, bytes=0)
    points = []
    for n_pf in SWEEP5["n_pf"]:
        for T in SWEEP5["T"]:
            for alpha in SWEEP5["alpha"]:
                if max_points is not None and len(points) >= max_points:
                    break
                w = workload_config5(pool, ptok, n_pf, T, alpha, n_chains=256)
                d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits,
                                            tokens=w.tokens, V=w.V, alpha=w.alpha, tau=w.tau,
                                            max_steps=w.max_steps, row_index=w.row_index)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                with torch.cuda.stream(stream):
                    for _ in range(warmup):
                        d.step(stream)
                    ev[0].record(stream)
                    for _ in range(steps):
                        d.step(stream)
                    ev[1].record(stream)
                    ev[2].record(stream)
                    for _ in range(steps):
                        d.score_rows(stream)
                    ev[3].record(stream)
                torch.cuda.synchronize()
                st = int(d.t["status"].item()) | int(d.t["wstatus"].item())
                assert st == 0, ps.dev_status_names(st)
                ms = ev[0].elapsed_time(ev[1]) / steps
                k1 = ev[2].elapsed_time(ev[3]) / steps
                units = w.layout.suffix_tokens()
                nbytes = w.n_rows * w.V * 2
                tot["tokens"] += units
                tot["rows"] += w.n_rows
                tot["ms"] += ms
                tot["k1_ms"] += k1
                tot["bytes"] += nbytes
                pt = {"n_pf": n_pf, "T": T, "alpha": alpha, "rows": w.n_rows,
                      "suffix_tokens": units, "ms_per_step": ms,
                      "tokens_per_s": units / ms * 1e3, "k1_ms": k1,
                      "logits_GBps": nbytes / k1 / 1e6}
                points.append(pt)
                if per_point:
                    print(json.dumps({"sweep_point": pt}), flush=True)
                del d, w
    del pool, ptok
    torch.cuda.empty_cache()
    rates = [p["tokens_per_s"] for p in points]
    gbps = [p["logits_GBps"] for p in points]
    return {"points": len(points), "n_chains": 256,
            "pool_rows": n_pool, "pool_bytes": n_pool * SWEEP5["V"] * 2, "l2_bytes": l2,
            "tokens_per_s": tot["tokens"] / tot["ms"] * 1e3,
            "rows": tot["rows"], "suffix_tokens": tot["tokens"],
            "logits_GBps": tot["bytes"] / tot["k1_ms"] / 1e6,
            "frac_of_8TBps": tot["bytes"] / tot["k1_ms"] / 1e6 / NOMINAL_HBM_GBS,
            "tokens_per_s_range": [min(rates), max(rates)],
            "logits_GBps_range": [min(gbps), max(gbps)],
            "steps_per_point": steps,
            "note": "each point's step and scoring kernel timed alone; totals over all points"}


def sweep(args) -> int:
    """--sweep: the throughput sweep alone, one JSON line per point and one
    with the aggregate (the default bench line carries the aggregate too)."""
    import __graft_entry__
    __graft_entry__.build()
    import mh_prefetch_subtree_gb300 as ps
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    agg = sweep_leg(ps, dev, stream, args.sweep_steps, max(1, args.sweep_warmup), per_point=True,
                    max_points=args.sweep_points)
    print(json.dumps({"sweep": agg}), flush=True)
    return 0


def steady_state_leg(ps, w, d, dev, stream, steps: int, warmup: int) -> dict:
    """The same round as the timed step, with the current state's per-position
    values carried from the previous round (the pages keep them; ps_carry_state
    produces them) instead of its rows scored again: the step scores only the
    requests' rows (through a row index into the same logits), assembles with
    the carried values, walks, and carries the reached state forward.
    Informative; the bench line scores the root rows."""
    import copy
    from synth.trees import assemble_layout
    lay = w.layout
    T = lay.T
    trees = [copy.deepcopy(t) for t in lay.trees]
    for t in trees:
        t.finalize_root_cut(T)                   # no root rows
    lay2 = assemble_layout(trees)
    keep, root_lp0, root_lq = [], [], []
    lp0_h, lq_h = d.t["lp0"].cpu().numpy(), d.t["lq"].cpu().numpy()
    for c in range(lay.n_chains):
        s0, s1 = int(lay.chain_seg0[c]), int(lay.chain_seg0[c + 1])
        r0, r1 = int(lay.seg_row0[s0]), int(lay.seg_row0[s0 + 1])
        rc = int(lay.seg_cut[s0])
        vals0, valsq = np.zeros(T), np.zeros(T)   # positions <= rc: earlier rounds' values
        vals0[rc:], valsq[rc:] = lp0_h[r0:r1], lq_h[r0:r1]
        root_lp0.append(vals0)
        root_lq.append(valsq)
        keep.extend(range(int(lay.seg_row0[s0 + 1]), int(lay.seg_row0[s1])))
    assert len(keep) == lay2.n_rows
    ri = torch.tensor(keep, dtype=torch.int64, device=dev)
    rl0 = torch.tensor(np.stack(root_lp0), dtype=torch.float64, device=dev)
    rlq = torch.tensor(np.stack(root_lq), dtype=torch.float64, device=dev)
    d2 = ps.DeviceSubtree.create(layout=lay2, u=w.u, logits=w.logits, tokens=w.tokens[ri],
                                 V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                 row_index=ri, root_lp0=rl0, root_lq=rlq)
    nxt = {k: torch.empty((lay.n_chains, T), dtype=torch.float64, device=dev) for k in ("lp0", "lq")}
    cst = torch.zeros(1, dtype=torch.int32, device=dev)
    io = ps.make_carry_io(state_seg=d2.t["state_seg"], row_lp0=d2.t["lp0"], row_lq=d2.t["lq"],
                          prev_lp0=rl0, prev_lq=rlq, next_lp0=nxt["lp0"], next_lq=nxt["lq"],
                          status=cst)

    def one():
        d2.step(stream)
        ps.ps_carry_state(d2.batch, io, stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            one()
        b.record(stream)
    torch.cuda.synchronize()
    st = int(d2.t["status"].item()) | int(d2.t["wstatus"].item()) | int(cst.item())
    assert st == 0, ps.dev_status_names(st)
    # the same log A as the step that scored the root rows
    req = ~lay.is_root()
    dla = np.abs(d2.t["log_accept"].cpu().numpy()[req] - d.t["log_accept"].cpu().numpy()[req])
    assert float(dla.max()) <= 1e-4, float(dla.max())
    ms = a.elapsed_time(b) / steps
    units = lay.suffix_tokens()
    return {"ms_per_step": ms, "value": units / (ms / 1e3), "unit": UNIT,
            "rows_scored": lay2.n_rows, "max_abs_dlogA_vs_step": float(dla.max()),
            "step": "score (requests' rows), suffix sums with carried root values and walk "
                    "in one call, then carry"}


def graph_leg(d, stream, steps: int, units: int) -> dict:
    """The same round captured once in a CUDA graph and replayed `steps` times:
    what the step costs without the host-side work of each call (informative;
    it matters for small batches, where that work is a large share)."""
    with torch.cuda.stream(stream):
        d.step(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        d.step(stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    ms = kernel_loop(stream, steps, g.replay)
    return {"ms_per_step": ms, "value": units / (ms / 1e3), "unit": UNIT,
            "how": "ps_score_walk_subtree captured in one CUDA graph, replayed back to back"}


def host_tree_timing(ps, T: int, n_pf: int, reps: int = 200) -> dict:
    """Host-side tree construction (ps_build_bfs_tree, ps_predictive_allocation)
    per call through the binding, for the bench's T and request budget.  The
    predictive allocation runs on a complete binary candidate tree of depth 8
    (511 nodes) with eq. (14) branch probabilities from seeded class
    probabilities and the pages' default budget of 20."""
    rng = np.random.default_rng(10086)
    cuts = rng.integers(0, T, 8 * n_pf).astype(np.int32)
    t0 = time.perf_counter()
    for _ in range(reps):
        ps.ps_build_bfs_tree(T, n_pf, None, cuts)
    bfs_us = (time.perf_counter() - t0) / reps * 1e6
    n = 511
    acc = np.array([2 * v + 1 if 2 * v + 1 < n else -1 for v in range(n)], np.int32)
    rej = np.array([2 * v + 2 if 2 * v + 2 < n else -1 for v in range(n)], np.int32)
    pa, pr = rng.uniform(0, 0.6, n), rng.uniform(0, 0.4, n)
    h = np.array([ps.ps_midpoint_branch_probability(a, r) for a, r in zip(pa, pr)])
    cand = np.ones(n, np.uint8)
    t0 = time.perf_counter()
    for _ in range(reps // 10):
        ps.ps_predictive_allocation(acc, rej, cand, h, 20)
    dp_us = (time.perf_counter() - t0) / (reps // 10) * 1e6
    return {"bfs_us": bfs_us, "bfs": f"T={T}, N_pf={n_pf}",
            "dp_us": dp_us, "dp": "511-node candidate tree, budget 20",
            "where": "host, per call through the binding"}


def kernel_loop(stream, steps: int, fn) -> float:
    """Average device time (ms) of fn() over `steps` back-to-back calls on
    `stream`, from CUDA events recorded on that stream."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def tail_after_scoring(d, stream, reps: int = 7, loop_ms: float = 250.0) -> dict:
    """What a round adds after its scoring kernel: rounds and scoring-kernel
    launches timed in alternating back-to-back loops of the same length, the
    median of the per-repetition differences.  Interleaving keeps slow drifts
    of the read rate out of the difference."""
    k1 = kernel_loop(stream, 3, lambda: d.score_rows(stream))
    n = max(20, min(2000, int(loop_ms / max(k1, 1e-3))))
    diffs = []
    for _ in range(reps):
        r = kernel_loop(stream, n, lambda: d.step(stream))
        k = kernel_loop(stream, n, lambda: d.score_rows(stream))
        diffs.append((r - k) * 1e3)
    return {"median_us": float(np.median(diffs)), "min_us": float(min(diffs)),
            "max_us": float(max(diffs)), "reps": reps, "rounds_per_loop": n}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="libps", choices=["libps", "reference"])
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave the 36-point throughput sweep out of the bench line")
    ap.add_argument("--no-extras", action="store_true",
                    help="time only the step and the scoring kernel (for profiling runs)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the round captured in a CUDA graph and replayed")
    ap.add_argument("--sweep", action="store_true",
                    help="time the 36-point throughput sweep alone, one line per point")
    ap.add_argument("--sweep-steps", type=int, default=2)
    ap.add_argument("--sweep-warmup", type=int, default=3)
    ap.add_argument("--sweep-points", type=int, default=None,
                    help="with --sweep: time only the first K points (for profiling runs)")
    ap.add_argument("--n-pf", type=int, default=None,
                    help="override the request budget (smaller batches for profiling)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    ws, rank, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, ws, rank)
    if args.sweep:
        return sweep(args) if rank == 0 else 0

    import __graft_entry__
    __graft_entry__.build()
    import mh_prefetch_subtree_gb300 as ps

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = build_workload(args.config, dev, rank, args.n_pf)
    lay = w.layout
    d = ps.DeviceSubtree.create(layout=lay, u=w.u, logits=w.logits, tokens=w.tokens, V=w.V,
                                alpha=w.alpha, tau=w.tau, max_steps=w.max_steps,
                                row_index=w.row_index, per_row=True, sums=True)
    stream = torch.cuda.Stream(device=dev)
    units_per_step = lay.suffix_tokens()
    rows = w.n_rows
    logits_bytes = w.logits_bytes()
    alg_bytes_k1 = rows * (w.V * w.elem_bytes + 4 + 16)   # logits + token in, lp0/lq out

    def step():
        d.step(stream)                  # ps_score_walk_subtree: scoring, sums and walk

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    st = int(d.t["status"].item()) | int(d.t["wstatus"].item())
    assert st == 0, ps.dev_status_names(st)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    with torch.cuda.stream(stream):
        # the timed steps: nothing is recorded between the kernels of a step, so
        # each kernel's launch overlaps the tail of the one before it
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
    torch.cuda.synchronize()
    # the scoring kernel alone, back to back on the same stream, for its roofline
    k1_avg = kernel_loop(stream, args.steps, lambda: d.score_rows(stream))
    clocks.mark(False)
    if ws > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), dev)
    st = int(d.t["status"].item()) | int(d.t["wstatus"].item())
    assert st == 0, ps.dev_status_names(st)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(units_per_step, ws, args.steps, total_ms)

    extras = {}
    if not args.no_extras:
        extras = variant_legs(ps, w, d, dev, stream, args.steps, logits_bytes)
        n_ch, T = lay.n_chains, lay.T
        extras["tree_construction"] = host_tree_timing(ps, T, int(w.info.get("n_requests", 16)))
        if args.graph:
            extras["graph_replay"] = graph_leg(d, stream, args.steps, units_per_step)
        if ws == 1 and getattr(w.layout, "trees", None):
            extras["steady_state"] = steady_state_leg(ps, w, d, dev, stream, args.steps,
                                                      args.warmup)
    # after the variant legs, so that a launch list of the first launches
    # still holds one of each kernel
    tail = tail_after_scoring(d, stream)
    clocks.stop()

    # ---- end to end through the public API, host buffers ------------------
    e2e = None
    if not args.no_e2e:
        # every rank on this host pins its own copy of the batch's inputs; if
        # the host cannot hold them all, no rank runs the leg (it has barriers)
        need = logits_bytes + rows * 4 + (1 << 30)
        local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", str(ws)))
        avail = host_memory_available()
        short = 1.0 if avail is not None and avail < local_ranks * need * 1.25 + (8 << 30) else 0.0
        if max_over_ranks(short, dev) > 0:
            e2e = {"skipped": f"pinning {local_ranks} x {need / 1e9:.1f} GB of inputs would "
                              f"exceed the host's available memory ({(avail or 0) / 1e9:.0f} GB)"}
        else:
            e2e = e2e_leg(ps, w, d, dev, stream, args, ws)

    peak, peak_src = peaks()
    achieved = alg_bytes_k1 / (k1_avg / 1e3) / 1e9
    traffic = None
    if (NCU_TRAFFIC["source_sha1"] == kernel_source_sha1() and args.config == NCU_TRAFFIC["config"]
            and args.n_pf is None):
        traffic = NCU_TRAFFIC["bytes_per_launch"]     # captured on this workload
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        # the arithmetic: float32 exponent sums per row, float64 per-row finish
        # and suffix sums; the logits themselves are stored as config.logits_dtype
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded logits, trees of the configuration's rule, proposal tokens "
                "drawn from q_tau)",
        "config": {"workload": w.name, "V": w.V, "T": lay.T, "n_requests": lay.n_seg - lay.n_chains,
                   "rows": rows, "suffix_tokens": units_per_step, "logits_bytes": logits_bytes,
                   "logits_dtype": w.dtype,
                   "alpha": w.alpha, "tau": w.tau,
                   "l2": f"inputs {logits_bytes / 1e9:.1f} GB > 129 MB L2; no flush",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} hbm_gbs (a read+write copy; a read-only "
                                    "stream can exceed it)",
                     "kernel": "score_rows_tail_kernel", "kernel_ms": k1_avg,
                     "algorithmic_bytes": alg_bytes_k1,
                     "frac_of_8TBps": achieved / NOMINAL_HBM_GBS},
        "logits_GBps": logits_bytes / (k1_avg / 1e3) / 1e9,
        "rows_per_s": whole_job_rate(rows, ws, args.steps, total_ms),
        "gpu_launches": 2 * args.steps,
        "kernel_launches_per_step": {"score_rows_tail_kernel (scoring)": 1,
                                     "assemble_kernel (suffix sums, log A and the walk)": 1},
        # what the suffix sums, log A and the walk add to a step after scoring
        "after_scoring_us": tail["median_us"],
        "after_scoring": dict(tail, how="median over alternating loops of rounds and of the "
                                        "scoring kernel alone"),
        "clocks": clocks.summary(),
    }
    line.update(extras)
    if "read_probe" in line:
        line["read_probe"]["scoring_kernel_ratio"] = line["logits_GBps"] / line["read_probe"]["GBps"]
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        ref, line["cpu_baseline"] = cpu_baseline(w)
        line["parity"] = parity_vs_oracle(w, d, ref)
    if rank == 0 and ws == 1 and not args.no_sweep:
        del d, w
        torch.cuda.empty_cache()
        line["sweep"] = sweep_leg(ps, dev, stream, args.sweep_steps, args.sweep_warmup)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def variant_legs(ps, w, d, dev, stream, steps: int, logits_bytes: int) -> dict:
    """The scoring kernel's other variants on the same batch, each timed back
    to back on the bench stream: with the entropy of p0, at three temperatures
    in one pass, at a temperature whose 1/tau is not an integer (a second
    exponential per logit), that with the entropy; and the round carry-over."""
    n = w.n_rows
    f64 = lambda *shape: torch.empty(shape, dtype=torch.float64, device=dev)
    ent_rows, lp0_v, lq_v = f64(n), f64(n), f64(n)
    mt_taus = [0.25, 0.5, 1.0]          # MultiTryMH candidate temperatures
    mt_lq = f64(len(mt_taus), n)
    bg = type(d.batch).from_buffer_copy(d.batch)
    bg.tau = GENERAL_TAU
    bg._keep = d.batch._keep
    rate = lambda ms: {"kernel_ms": ms, "logits_GBps": logits_bytes / (ms / 1e3) / 1e9,
                       "frac_of_8TBps": logits_bytes / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS}
    out = {}
    out["with_entropy"] = rate(kernel_loop(stream, steps, lambda: ps.ps_score_rows(
        d.batch, lp0_v, lq_v, d.t["status"], d.workspace, stream, entropy=ent_rows)))
    out["multi_temperature"] = dict(taus=mt_taus, **rate(kernel_loop(
        stream, steps, lambda: ps.ps_score_rows_multi(d.batch, mt_taus, lp0_v, mt_lq,
                                                      d.t["status"], d.workspace, stream))))
    out["general_tau"] = dict(tau=GENERAL_TAU, **rate(kernel_loop(
        stream, steps, lambda: ps.ps_score_rows(bg, lp0_v, lq_v, d.t["status"], d.workspace,
                                                stream))))
    out["general_tau_with_entropy"] = dict(tau=GENERAL_TAU, **rate(kernel_loop(
        stream, steps, lambda: ps.ps_score_rows(bg, lp0_v, lq_v, d.t["status"], d.workspace,
                                                stream, entropy=ent_rows))))
    st = int(d.t["status"].item())
    assert st == 0, ps.dev_status_names(st)
    # a masked vocabulary (all but the first 1000 ids at -inf, tokens among
    # them) in the entropy variant, without and with the masked-logits hint
    masked = w.logits.clone()
    masked[:, 1000:] = float("-inf")
    mtok = (w.tokens % 1000).to(torch.int32)
    mb = {flags: ps.make_batch(V=w.V, T=w.layout.T, alpha=w.alpha, tau=w.tau,
                               chain_seg0=d.t["chain_seg0"], seg_row0=d.t["seg_row0"],
                               seg_cut=d.t["seg_cut"], seg_src=d.t["seg_src"], logits=masked,
                               tokens=mtok, flags=flags)
          for flags in (0, ps.PS_FLAG_MASKED_LOGITS)}
    out["masked_vocabulary_with_entropy"] = {
        "no_hint": rate(kernel_loop(stream, steps, lambda: ps.ps_score_rows(
            mb[0], lp0_v, lq_v, d.t["status"], d.workspace, stream, entropy=ent_rows))),
        "masked_logits_hint": rate(kernel_loop(stream, steps, lambda: ps.ps_score_rows(
            mb[ps.PS_FLAG_MASKED_LOGITS], lp0_v, lq_v, d.t["status"], d.workspace, stream,
            entropy=ent_rows))),
        "vocabulary": "all but the first 1000 ids at -inf"}
    del masked, mb
    st = int(d.t["status"].item())
    assert st == 0, ps.dev_status_names(st)
    # the kernels after scoring on their own (the round runs them as one
    # kernel): ps_assemble_subtree and ps_walk_subtree back to back
    out["after_scoring_kernels_alone"] = {
        "suffix_sums_us": kernel_loop(stream, steps, lambda: d.assemble(stream)) * 1e3,
        "walk_us": kernel_loop(stream, steps, lambda: d.walk(stream)) * 1e3}
    # a plain streaming read of the same logits buffer on the same box: the
    # read rate the scoring kernel's own rate is compared with
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    read_ms = kernel_loop(stream, steps, lambda: ps.ps_selftest_read(w.logits, sink, stream))
    read_bytes = w.logits.numel() * w.logits.element_size()
    out["read_probe"] = {"kernel_ms": read_ms, "GBps": read_bytes / (read_ms / 1e3) / 1e9,
                         "bytes": read_bytes,
                         "how": "ps_selftest_read: 16-byte streaming loads, 8 in flight per "
                                "thread, 4 x 512 threads per SM, over the batch's logits"}
    # the round carry-over (reached state's per-position values) after a step
    lay = w.layout
    n_ch, T = lay.n_chains, lay.T
    cy_out = {k: f64(n_ch, T) for k in ("lp0", "lq")}
    cy_prev = {k: torch.zeros((n_ch, T), dtype=torch.float64, device=dev) for k in ("lp0", "lq")}
    cy_ll = f64(n_ch)
    cy_status = torch.zeros(1, dtype=torch.int32, device=dev)
    io = ps.make_carry_io(state_seg=d.t["state_seg"], row_lp0=d.t["lp0"], row_lq=d.t["lq"],
                          prev_lp0=cy_prev["lp0"], prev_lq=cy_prev["lq"],
                          next_lp0=cy_out["lp0"], next_lq=cy_out["lq"], loglik=cy_ll,
                          status=cy_status)
    carry_ms = kernel_loop(stream, steps, lambda: ps.ps_carry_state(d.batch, io, stream))
    assert int(cy_status.item()) == 0, ps.dev_status_names(int(cy_status.item()))
    out["carry"] = {"kernel_ms": carry_ms, "GBps": n_ch * T * 32 / (carry_ms / 1e3) / 1e9,
                    "bytes": "per position: 16 B read (row or previous value), 16 B written"}
    return out


def e2e_leg(ps, w, d, dev, stream, args, ws, chunks: int = 8):
    """Same metric through the public API with the batch's inputs in pinned host
    memory and its results read back, every step.

    The host-to-device copies of the logits and tokens are split into row
    chunks on a copy stream; ps_score_rows scores each chunk as soon as it has
    landed (the per-row scores of a chunk are independent), then
    ps_assemble_subtree and ps_walk_subtree run and log A and the walk's
    results are copied back.
    """
    lay = w.layout
    h = {}
    h["logits"] = torch.empty(w.logits.shape, dtype=w.logits.dtype, pin_memory=True)
    h["logits"].copy_(w.logits)
    h["tokens"] = w.tokens.cpu().pin_memory()
    meta = {k: d.t[k] for k in ("chain_seg0", "seg_row0", "seg_cut", "seg_src", "chain_node0",
                                "acc", "rej", "req", "u")}
    hmeta = {k: v.cpu().pin_memory() for k, v in meta.items()}
    outs = {k: d.t[k] for k in ("log_accept", "state_seg", "end_node", "k_delta", "path")}
    hout = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = (h["logits"].numel() * h["logits"].element_size() + h["tokens"].numel() * 4
           + sum(v.numel() * v.element_size() for v in hmeta.values()))
    d2h = sum(v.numel() * v.element_size() for v in hout.values())
    n = w.n_rows
    bounds = [n * i // chunks for i in range(chunks + 1)]
    subs = []
    for i in range(chunks):
        r0, r1 = bounds[i], bounds[i + 1]
        if r1 == r0:
            continue
        b = ps.make_batch(V=w.V, T=lay.T, alpha=w.alpha, tau=w.tau,
                          chain_seg0=d.t["chain_seg0"], seg_row0=d.t["seg_row0"],
                          seg_cut=d.t["seg_cut"], seg_src=d.t["seg_src"],
                          logits=w.logits[r0:r1], tokens=w.tokens[r0:r1], n_rows=r1 - r0)
        subs.append((r0, r1, b, d.t["lp0"][r0:r1], d.t["lq"][r0:r1]))
    copy = torch.cuda.Stream(device=dev)
    landed = [torch.cuda.Event() for _ in subs]
    start_ev = torch.cuda.Event()

    def step():
        start_ev.record(stream)
        copy.wait_event(start_ev)
        with torch.cuda.stream(copy):
            for k, v in meta.items():
                v.copy_(hmeta[k], non_blocking=True)
            for (r0, r1, _, _, _), ev in zip(subs, landed):
                w.logits[r0:r1].copy_(h["logits"][r0:r1], non_blocking=True)
                w.tokens[r0:r1].copy_(h["tokens"][r0:r1], non_blocking=True)
                ev.record(copy)
        d.t["status"].zero_()
        d.t["wstatus"].zero_()
        for (r0, r1, b, lp0, lq), ev in zip(subs, landed):
            stream.wait_event(ev)
            ps.ps_score_rows(b, lp0, lq, d.t["status"], d.workspace, stream)  # no entropy
        d.assemble(stream)
        d.walk(stream)
        for k, v in outs.items():
            hout[k].copy_(v, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    st = int(d.t["status"].item()) | int(d.t["wstatus"].item())
    assert st == 0, ps.dev_status_names(st)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_steps = args.e2e_steps
    if ws > 1:
        torch.distributed.barrier()
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(n_steps):
            step()
        b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), dev)
    v = whole_job_rate(lay.suffix_tokens(), ws, n_steps, ms)
    return {"value": v, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n_steps, "ms_per_step": ms / n_steps,
            "h2d_GBps": h2d / (ms / 1e3 / n_steps) / 1e9, "row_chunks": len(subs)}


if __name__ == "__main__":
    sys.exit(main())
