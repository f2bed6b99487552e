"""CPU oracle for scoring one prefetched subtree batch and walking it.

TEST INFRASTRUCTURE.  Only the tests, the package's ``smoke()`` check and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never calls it.

It is written from "PreSTO: Predictive Subtree Prefetching for Fast LLM Power
Sampling" (arXiv 2610.13171) in float64, step by step and without shortcuts:

* ``row_logprobs``      per-token log p0 and log q_tau from the same logits
                        (Appendix B.1, last paragraph; Appendix D.3), in C;
                        called once per temperature it is also the oracle of
                        multi-temperature scoring (MultiTryMH, Table 6(a));
* ``materialize``       the full state of every tree node as an explicit
                        position -> row map (section 3.2 step (1); a rejection
                        child keeps its parent's state; Condition 1);
* ``suffix_sums``       log p0 / log q_tau of the y and x suffixes by summing
                        token log-probabilities over positions c+1..T
                        (eq. (6), Appendix B.1 eq. (7)-(9)), optionally with the
                        current state's values carried from the previous round;
* ``carry_state``       the reached state's per-position values for the next
                        round, with eq. (21) log-likelihood and eq. (22)
                        confidence (section 3.2 step (3));
* ``log_accept``        log A = min{0, log q(x|y) - log q(y|x) + alpha (log p0(y) - log p0(x))}
                        (eq. (6));
* ``walk``              the MH walk over the subtree: accept iff u <= A, left
                        on accept, right on reject, stop at a leaf, a deferred
                        node or after K - k transitions (section 3.2 step (3),
                        Example 5, Algorithm 2);
* ``replay``            sequential PowerMH on explicit states with the same
                        uniforms (Proposition 1);
* ``expected_transitions``  F_I(v0) = sum of reaching weights (Lemma 1, eq. (11)-(12));
* ``eps_class``, ``eps_certain_fraction``  epsilon-certainty of each decision
                        and their share (section 3.3);
* entropy of p0 per row (``row_logprobs(..., entropy=True)``; Appendix D.3).

Every function is pinned by the ``-m "not gpu"`` tests against closed forms,
library routines, brute force or the pages' worked examples.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(HERE, "_build")
_SO = os.path.join(_BUILD, "libps_oracle.so")
_SRC = os.path.join(HERE, "ps_oracle.c")

LEAF = -1
DEFERRED = -2


def build(force: bool = False) -> str:
    """Compile the C part of the oracle with gcc (fp64, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.oracle_row_logprobs.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        L.oracle_row_logprobs.restype = None
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def default_threads() -> int:
    return int(os.environ.get("PS_ORACLE_THREADS", os.cpu_count() or 1))


def row_logprobs(logits: np.ndarray, dtype: str, V: int, tokens: np.ndarray,
                 tau: float, row_index: np.ndarray | None = None,
                 threads: int | None = None, entropy: bool = False):
    """Per-row (lp0, lq) in float64, and the entropy of p0 when entropy=True
    (then a third array is returned).

    ``logits`` is a 2-D array [n_logit_rows, ld]: uint16 holding bf16 bit
    patterns (dtype "bf16") or float32 (dtype "f32").  Row r reads logits row
    row_index[r] (identity when None) and token tokens[r].
    """
    if dtype == "bf16":
        assert logits.dtype == np.uint16
        dcode = 0
    elif dtype == "f32":
        assert logits.dtype == np.float32
        dcode = 1
    else:
        raise ValueError(dtype)
    logits = np.ascontiguousarray(logits)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    ld = logits.shape[1]
    assert V <= ld
    ri = None
    if row_index is not None:
        ri = np.ascontiguousarray(row_index, dtype=np.int64)
        assert ri.shape[0] == n
        assert n == 0 or (ri.min() >= 0 and ri.max() < logits.shape[0])
    else:
        assert logits.shape[0] >= n
    lp0 = np.empty(n, dtype=np.float64)
    lq = np.empty(n, dtype=np.float64)
    ent = np.empty(n, dtype=np.float64) if entropy else None
    lib().oracle_row_logprobs(
        logits.ctypes.data, dcode, int(V), int(ld), int(n),
        None if ri is None else ri.ctypes.data, tokens.ctypes.data, float(tau),
        lp0.ctypes.data, lq.ctypes.data, None if ent is None else ent.ctypes.data,
        int(threads or default_threads()))
    if entropy:
        return lp0, lq, ent
    return lp0, lq


# ---------------------------------------------------------------------------
# States, sums, log A (eq. (6)), walk (section 3.2 step (3)), replay (Prop. 1)
# ---------------------------------------------------------------------------

@dataclass
class ChainStates:
    """Explicit state of every node of one chain.

    ``rows[v]`` is an int64 array of length T+1: rows[v][t] is the global row
    whose logits score position t of node v's state (index 0 unused), or -1
    for a position of the current state below the root segment (never scored).
    ``rows[v]`` is None for a deferred acceptance child (not generated).
    """

    T: int
    root_seg: int
    rows: list
    state_seg: list     # segment whose proposal the node's state came from


def materialize(layout, c: int) -> ChainStates:
    """Build every node's state of chain c by walking the tree from the root.

    The root holds the current state x (root segment rows for positions
    > root cut).  Expanding a node v with feasible request s of cut c_s gives
    the acceptance child the state (state(v)_{0:c_s}, y^s_{c_s+1:T}) and the
    rejection child a copy of state(v) (section 3.2 step (1)).  Condition 1 is
    checked as its consequence: the prefix a request conditions on,
    state(v)_{0:c_s}, must equal the root's prefix, which is all that exists
    when the batch is generated.
    """
    T = layout.T
    s0, s1 = int(layout.chain_seg0[c]), int(layout.chain_seg0[c + 1])
    n0, n1 = int(layout.chain_node0[c]), int(layout.chain_node0[c + 1])
    root = s0
    rc = int(layout.seg_cut[root])
    r0 = int(layout.seg_row0[root])
    assert int(layout.seg_row0[root + 1]) - r0 == T - rc
    base = np.full(T + 1, -1, dtype=np.int64)
    base[rc + 1:] = r0 + np.arange(T - rc, dtype=np.int64)
    nn = n1 - n0
    rows = [None] * nn
    state_seg = [None] * nn
    rows[0] = base
    state_seg[0] = root
    order = [0]
    for v in order:                      # parents before children
        if rows[v] is None:
            continue
        a = int(layout.acc[n0 + v])
        b = int(layout.rej[n0 + v])
        s = int(layout.req[n0 + v])
        if b >= 0:
            rows[b - n0] = rows[v].copy()
            state_seg[b - n0] = state_seg[v]
            order.append(b - n0)
        if s >= 0:
            assert s0 <= s < s1 and s != root
            cs = int(layout.seg_cut[s])
            assert 0 <= cs <= T - 1
            assert np.array_equal(rows[v][1:cs + 1], base[1:cs + 1]), \
                "Condition 1 violated: the request's prefix is not the root's"
            rs = int(layout.seg_row0[s])
            assert int(layout.seg_row0[s + 1]) - rs == T - cs
            new = rows[v].copy()
            new[cs + 1:] = rs + np.arange(T - cs, dtype=np.int64)
            rows[a - n0] = new
            state_seg[a - n0] = s
            order.append(a - n0)
        elif a >= 0:
            state_seg[a - n0] = None      # deferred or unexpanded acceptance child
    return ChainStates(T=T, root_seg=root, rows=rows, state_seg=state_seg)


def _pos_values(st_rows, c, row_vals, root_vals, T, t0=1):
    """Values of positions t0..T of one state (index t of the returned array is
    position t): the row value where the state has a scored row, else the
    chain root's carried value for that position."""
    out = np.full(T + 1, np.nan)
    rows = np.asarray(st_rows[t0:T + 1], dtype=np.int64)
    has = rows >= 0
    vals = np.asarray(row_vals)[np.where(has, rows, 0)]
    if not has.all():
        assert root_vals is not None, "root position without a row or a carried value"
        vals = np.where(has, vals, np.asarray(root_vals)[c, t0 - 1:T])
    out[t0:] = vals
    return out


def suffix_sums(layout, lp0: np.ndarray, lq: np.ndarray, states=None,
                root_lp0: np.ndarray | None = None, root_lq: np.ndarray | None = None) -> dict:
    """LP_y, LQ_y, LP_x, LQ_x for every request (NaN at chain roots).

    For the request s issued at node v with cut c_s: the y suffix is positions
    c_s+1..T of the acceptance child's state, the x suffix the same positions of
    state(v); each sum adds token log-probabilities (eq. (6) and the sum under it).
    Positions of the current state that have no scored row take the values the
    previous round retained (root_lp0/root_lq [n_chains, T], position t at
    column t-1; section 3.2 step (3)).
    """
    n = layout.n_seg
    out = {k: np.full(n, np.nan) for k in ("lp_y", "lq_y", "lp_x", "lq_x")}
    T = layout.T
    for c in range(layout.n_chains):
        st = materialize(layout, c) if states is None else states[c]
        n0, n1 = int(layout.chain_node0[c]), int(layout.chain_node0[c + 1])
        for v in range(n1 - n0):
            s = int(layout.req[n0 + v])
            if s < 0 or st.rows[v] is None:
                continue
            cs = int(layout.seg_cut[s])
            a = int(layout.acc[n0 + v]) - n0
            vy0 = _pos_values(st.rows[a], c, lp0, root_lp0, T, cs + 1)
            vyq = _pos_values(st.rows[a], c, lq, root_lq, T, cs + 1)
            vx0 = _pos_values(st.rows[v], c, lp0, root_lp0, T, cs + 1)
            vxq = _pos_values(st.rows[v], c, lq, root_lq, T, cs + 1)
            out["lp_y"][s] = np.sum(vy0[cs + 1:])
            out["lq_y"][s] = np.sum(vyq[cs + 1:])
            out["lp_x"][s] = np.sum(vx0[cs + 1:])
            out["lq_x"][s] = np.sum(vxq[cs + 1:])
    return out


def carry_state(layout, state_seg: np.ndarray, row_vals: dict, prev: dict) -> dict:
    """The reached state's retained per-position values for the next round
    (section 3.2 step (3): the sampler keeps the token-level log-probabilities
    of the state it moves to), and the statistics of eq. (21) and (22).

    row_vals: per-row arrays of this batch, e.g. {"lp0": .., "lq": .., "entropy": ..};
    prev: the same keys, each [n_chains, T]: the values of the current state,
    used for positions below the root cut.  Returns [n_chains, T] arrays with
    the same keys, plus "loglik" = mean of lp0 over positions 1..T (eq. (21))
    and, when entropy is given, "confidence" = minus the mean entropy (eq. (22)).
    """
    T = layout.T
    nc = layout.n_chains
    out = {k: np.empty((nc, T)) for k in row_vals}
    for c in range(nc):
        st = materialize(layout, c)
        s = int(state_seg[c])
        # a node holding the reached state: any node whose state came from s
        v = next(i for i, x in enumerate(st.state_seg) if x == s and st.rows[i] is not None)
        for k, vals in row_vals.items():
            pv = _pos_values(st.rows[v], c, vals, prev.get(k), T)
            out[k][c] = pv[1:]
    out["loglik"] = out["lp0"].mean(axis=1)
    if "entropy" in out:
        out["confidence"] = -out["entropy"].mean(axis=1)
    return out


def log_accept(sums: dict, alpha: float) -> tuple[np.ndarray, np.ndarray]:
    """eq. (6): r = log q_tau(x|.) - log q_tau(y|.) + alpha (log p0(y|.) - log p0(x|.)),
    log A = min{0, r}."""
    r = (sums["lq_x"] - sums["lq_y"]) + alpha * (sums["lp_y"] - sums["lp_x"])
    with np.errstate(invalid="ignore"):
        la = np.where(np.isnan(r), np.nan, np.minimum(0.0, r))
    return r, la


def walk(layout, logA: np.ndarray, u: np.ndarray, max_steps: int) -> dict:
    """MH transitions over each chain's subtree (section 3.2 step (3), Example 5).

    From the root, at each node whose request was scored: one transition;
    move to the acceptance child if u <= A (the accept test of Algorithm 1), else to the
    rejection child.  Stop at a leaf, at a node whose request was deferred, or
    after max_steps (= K - k) transitions.  The reached state is the segment
    of the last accepted proposal, or the root segment.
    """
    nc = layout.n_chains
    out = dict(state_seg=np.zeros(nc, np.int32), end_node=np.zeros(nc, np.int32),
               k_delta=np.zeros(nc, np.int32), path=[])
    for c in range(nc):
        v = int(layout.chain_node0[c])
        state = int(layout.chain_seg0[c])
        path = [v]
        k = 0
        while k < max_steps:
            s = int(layout.req[v])
            if s < 0:                     # LEAF or DEFERRED
                break
            A = np.exp(logA[s])
            k += 1
            if u[s] <= A:
                v = int(layout.acc[v])
                state = s
            else:
                v = int(layout.rej[v])
            path.append(v)
        out["state_seg"][c] = state
        out["end_node"][c] = v
        out["k_delta"][c] = k
        out["path"].append(path)
    return out


def replay(layout, lp0: np.ndarray, lq: np.ndarray, alpha: float, u: np.ndarray,
           max_steps: int) -> list:
    """Sequential PowerMH with the tree's random inputs (Proposition 1).

    The chain keeps its current state as an explicit position -> row map.  At
    each step the tree supplies the decision's random inputs (cut c, the
    proposal generated for that decision and its uniform u); the proposal
    y = (x_{0:c}, y_{c+1:T}) is formed from the *current sequential state*,
    A is computed from the two explicit sequences with eq. (6), and u <= A
    decides.  Returns, per chain, the list of states (row maps) after each
    committed transition k = 0..k_Delta, to compare with the walk.
    """
    res = []
    T = layout.T
    for c in range(layout.n_chains):
        st = materialize(layout, c)
        n0 = int(layout.chain_node0[c])
        x = st.rows[0].copy()
        base = st.rows[0]
        v = 0
        states = [x.copy()]
        k = 0
        while k < max_steps:
            s = int(layout.req[n0 + v])
            if s < 0:
                break
            cs = int(layout.seg_cut[s])
            # (A1): the proposal was generated from the root's prefix
            assert np.array_equal(x[1:cs + 1], base[1:cs + 1])
            rs = int(layout.seg_row0[s])
            y = x.copy()
            y[cs + 1:] = rs + np.arange(T - cs, dtype=np.int64)
            xs, ys = x[cs + 1:], y[cs + 1:]
            r = (lq[xs].sum() - lq[ys].sum()) + alpha * (lp0[ys].sum() - lp0[xs].sum())
            A = np.exp(min(0.0, r))
            k += 1
            if u[s] <= A:
                x = y
                v = int(layout.acc[n0 + v]) - n0
            else:
                v = int(layout.rej[n0 + v]) - n0
            states.append(x.copy())
        res.append(states)
    return res


def expected_transitions(layout, logA: np.ndarray, max_steps: int) -> np.ndarray:
    """E[k_Delta] per chain = sum of reaching weights over the scored decision
    nodes the walk can visit (Lemma 1, eq. (11)-(12), with h = A, epsilon = 0).

    A node counts when its own request was scored, every decision on its path
    from the root was scored, and its depth is below max_steps.
    """
    out = np.zeros(layout.n_chains)
    for c in range(layout.n_chains):
        n0 = int(layout.chain_node0[c])
        stack = [(n0, 1.0, 0)]
        tot = 0.0
        while stack:
            v, R, d = stack.pop()
            s = int(layout.req[v])
            if s < 0 or d >= max_steps:
                continue
            tot += R
            A = float(np.exp(logA[s]))
            stack.append((int(layout.acc[v]), R * A, d + 1))
            stack.append((int(layout.rej[v]), R * (1.0 - A), d + 1))
        out[c] = tot
    return out


def eps_class(logA: np.ndarray, eps: float = 0.01) -> np.ndarray:
    """epsilon-certainty class of each decision (section 3.3): 0 = certain
    reject (A <= eps), 2 = certain accept (A >= 1 - eps), 1 = uncertain;
    -1 where log A is NaN (chain roots)."""
    A = np.exp(logA)
    out = np.where(A <= eps, 0, np.where(A >= 1.0 - eps, 2, 1)).astype(np.int8)
    out[np.isnan(logA)] = -1
    return out


def eps_certain_fraction(logA: np.ndarray, eps: float = 0.01) -> float:
    """Share of scored decisions with A >= 1 - eps or A <= eps (section 3.3)."""
    a = np.exp(logA[~np.isnan(logA)])
    if a.size == 0:
        return float("nan")
    return float(np.mean((a >= 1.0 - eps) | (a <= eps)))


def score_subtree(logits: np.ndarray, dtype: str, V: int, tokens: np.ndarray,
                  layout, alpha: float, tau: float, row_index=None,
                  threads: int | None = None) -> dict:
    """Everything the scoring call returns, from the definitions above."""
    lp0, lq = row_logprobs(logits, dtype, V, tokens, tau, row_index, threads)
    sums = suffix_sums(layout, lp0, lq)
    r, la = log_accept(sums, alpha)
    out = dict(lp0=lp0, lq=lq, log_ratio=r, log_accept=la)
    out.update(sums)
    return out
