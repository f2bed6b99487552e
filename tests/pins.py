"""Pin checks for the oracle's assembly and walk, written as functions.

Each ``pin_*`` takes the oracle functions it checks as arguments, so the
planted-mistake tests can hand it a deliberately broken variant and show that
the pin fails.  The expected values come from the pages (Example 5, Condition
1, eq. (1)) and from closed forms, never from the oracle under test.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

from synth.trees import assemble_layout, bfs_tree, example5_tree

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f32_rows(n, V, fill):
    return np.full((n, V), fill, dtype=np.float32)


def pin_uniform_counts(row_logprobs, suffix_sums, T=12, V=50):
    """Uniform rows give -log V per token, so every suffix sum over positions
    c+1..T is exactly -(T - c) log V: catches a dropped or extra position."""
    rng = np.random.default_rng(11)
    lay = assemble_layout([bfs_tree(rng, T, 6)])
    n = lay.n_rows
    x = _f32_rows(n, V, 0.5)
    tok = rng.integers(0, V, n).astype(np.int32)
    lp0, lq = row_logprobs(x, "f32", V, tok, 0.25)
    sums = suffix_sums(lay, lp0, lq)
    req = ~lay.is_root()
    want = -(T - lay.seg_cut[req].astype(np.float64)) * math.log(V)
    for k in ("lp_y", "lq_y", "lp_x", "lq_x"):
        np.testing.assert_allclose(sums[k][req], want, rtol=1e-12)


def pin_mh_closed_form(row_logprobs, suffix_sums, log_accept, V=64, T=10):
    """With tau = 1 the proposal is p0 itself, and eq. (1) gives
    A = min{1, (p0(y)/p0(x))^(alpha-1)} directly.  x rows are uniform
    (p0 = 1/V per token), y rows put a margin of 40 on their token, so
    log A(x -> y) = min{0, (alpha-1) * n * (log V - eps)} = 0 and
    log A(y -> x) = -(alpha-1) * n * (log V - eps) with n = T - c and
    eps = log1p((V-1) e^-40).  Catches a sign error or a misplaced alpha."""
    alpha = 4.0
    eps = math.log1p((V - 1) * math.exp(-40.0))
    for y_peaked in (True, False):
        t = example5_tree(T, c1=3, c2=3)
        lay = assemble_layout([t])
        n = lay.n_rows
        x = np.zeros((n, V), dtype=np.float32)
        tok = np.zeros(n, dtype=np.int32)
        r0, r1 = int(lay.seg_row0[1]), int(lay.seg_row0[2])     # request y rows
        peak_rows = range(r0, r1) if y_peaked else range(0, int(lay.seg_row0[1]))
        for r in peak_rows:
            tok[r] = r % V
            x[r, tok[r]] = 40.0
        lp0, lq = row_logprobs(x, "f32", V, tok, 1.0)
        sums = suffix_sums(lay, lp0, lq)
        r, la = log_accept(sums, alpha)
        nn = T - int(lay.seg_cut[1])
        gain = (alpha - 1.0) * nn * (math.log(V) - eps)
        if y_peaked:
            np.testing.assert_allclose(r[1], gain, rtol=1e-12)
            assert la[1] == 0.0
        else:
            np.testing.assert_allclose(r[1], -gain, rtol=1e-12)
            np.testing.assert_allclose(la[1], -gain, rtol=1e-12)


def pin_alpha_tau_one(row_logprobs, suffix_sums, log_accept, V=300, T=40):
    """alpha = tau = 1: the target is p0 and so is the proposal, so every
    proposal is accepted: r = 0 for any logits and tokens (eq. (1))."""
    rng = np.random.default_rng(12)
    lay = assemble_layout([bfs_tree(rng, T, 8), bfs_tree(rng, T, 5)])
    n = lay.n_rows
    x = rng.normal(scale=3.0, size=(n, V)).astype(np.float32)
    tok = rng.integers(0, V, n).astype(np.int32)
    lp0, lq = row_logprobs(x, "f32", V, tok, 1.0)
    sums = suffix_sums(lay, lp0, lq)
    r, _ = log_accept(sums, 1.0)
    req = ~lay.is_root()
    scale = np.abs(sums["lp_x"][req]) + np.abs(sums["lp_y"][req])
    assert np.all(np.abs(r[req]) <= 1e-12 * scale + 1e-300)


def _copy_rows(x, tok, dst_rows, src_rows):
    x[dst_rows] = x[src_rows]
    tok[dst_rows] = tok[src_rows]


def pin_y_equals_x(row_logprobs, suffix_sums, log_accept, materialize, V=200, T=30):
    """A proposal whose suffix rows and tokens copy the from-state's gives
    log A = 0 exactly (eq. (6): both sums add the same numbers)."""
    rng = np.random.default_rng(13)
    lay = assemble_layout([bfs_tree(rng, T, 8)])
    n = lay.n_rows
    x = rng.normal(scale=3.0, size=(n, V)).astype(np.float32)
    tok = rng.integers(0, V, n).astype(np.int32)
    st = materialize(lay, 0)
    # copy in BFS order so that a from-state is final before it is copied
    for v in range(lay.n_nodes):
        s = int(lay.req[v])
        if s < 0:
            continue
        cs = int(lay.seg_cut[s])
        xs = st.rows[v][cs + 1:]
        ys = np.arange(int(lay.seg_row0[s]), int(lay.seg_row0[s + 1]))
        _copy_rows(x, tok, ys, xs)
    lp0, lq = row_logprobs(x, "f32", V, tok, 0.25)
    sums = suffix_sums(lay, lp0, lq)
    r, la = log_accept(sums, 4.0)
    req = ~lay.is_root()
    assert np.all(r[req] == 0.0) and np.all(la[req] == 0.0)


def pin_reversal(row_logprobs, suffix_sums, log_accept, V=128, T=20):
    """Reverse moves at the same cut: x -> y at v0 and y -> x at v1 (the second
    proposal copies x's suffix).  MH ratios of a move and its reverse are
    reciprocal, so r(x->y) + r(y->x) = 0 (eq. (7)-(9))."""
    rng = np.random.default_rng(14)
    for c in (0, 7, T - 1):
        t = example5_tree(T, c1=c, c2=c)
        lay = assemble_layout([t])
        n = lay.n_rows
        x = rng.normal(scale=2.0, size=(n, V)).astype(np.float32)
        tok = rng.integers(0, V, n).astype(np.int32)
        root = np.arange(int(lay.seg_row0[0]), int(lay.seg_row0[1]))
        rc = int(lay.seg_cut[0])
        xs = root[c - rc:]                        # root rows for positions c+1..T
        zs = np.arange(int(lay.seg_row0[2]), int(lay.seg_row0[3]))
        _copy_rows(x, tok, zs, xs)
        lp0, lq = row_logprobs(x, "f32", V, tok, 0.25)
        sums = suffix_sums(lay, lp0, lq)
        r, _ = log_accept(sums, 4.0)
        assert abs(r[1] + r[2]) <= 1e-12 * (abs(r[1]) + 1.0)
        assert r[1] != 0.0


def pin_two_segment_rule(materialize, n_trees=40):
    """Condition 1 makes every state x_{0:c_last} + y^last: the x suffix of
    request i is root rows (c_i, c_src] followed by the rows of src (section
    3.2, Condition 1; Figure 8(a)).  The full materialisation must agree."""
    rng = np.random.default_rng(15)
    for k in range(n_trees):
        T = int(rng.integers(2, 40))
        lay = assemble_layout([bfs_tree(rng, T, int(rng.integers(1, 12)))])
        st = materialize(lay, 0)
        rc = int(lay.seg_cut[0])
        r0 = int(lay.seg_row0[0])
        for v in range(lay.n_nodes):
            s = int(lay.req[v])
            if s < 0:
                continue
            ci = int(lay.seg_cut[s])
            src = int(lay.seg_src[s])
            csrc = T if src == 0 else int(lay.seg_cut[src])
            assert ci <= csrc                               # Condition 1
            want = list(range(r0 + ci - rc, r0 + csrc - rc))
            if src != 0:
                want += list(range(int(lay.seg_row0[src]), int(lay.seg_row0[src + 1])))
            assert list(st.rows[v][ci + 1:]) == want


def pin_rejection_inherits(materialize, n_trees=30):
    """A rejection child keeps its parent's state (section 3.2 step (1))."""
    rng = np.random.default_rng(16)
    for _ in range(n_trees):
        lay = assemble_layout([bfs_tree(rng, 25, 10)])
        st = materialize(lay, 0)
        for v in range(lay.n_nodes):
            b = int(lay.rej[v])
            if b >= 0 and st.rows[v] is not None:
                assert np.array_equal(st.rows[b], st.rows[v])
                assert st.state_seg[b] == st.state_seg[v]


def golden_example5():
    with open(os.path.join(GOLDEN, "example5_walk.json")) as f:
        return json.load(f)


def pin_example5(walk):
    """Example 5 (Appendix B.3): accept at v0, reject at v1 -> path v0, v1, v4,
    trajectory x -> y -> y, two transitions."""
    g = golden_example5()
    lay = assemble_layout([example5_tree(16, c1=9, c2=4)])
    name = {f"v{i}": i for i in range(5)}
    seg_of = {"x": 0, "y": 1, "z": 2}
    logA = np.array([np.nan, math.log(0.6), math.log(0.3)])
    # u <= A accepts (the accept test of Algorithm 1); choose u on the stated side
    u = np.ones(3)
    for node, dec in g["decisions"].items():
        s = int(lay.req[name[node]])
        A = math.exp(logA[s])
        u[s] = A * 0.5 if dec == "accept" else (1.0 + A) * 0.5
    out = walk(lay, logA, u, max_steps=100)
    assert out["path"][0] == [name[v] for v in g["expected_path"]]
    assert int(out["k_delta"][0]) == g["expected_k_delta"]
    assert int(out["state_seg"][0]) == seg_of[g["expected_trajectory"][-1]]
    assert int(out["end_node"][0]) == name[g["expected_path"][-1]]


def pin_library_log_softmax(row_logprobs, V=257):
    """Small random rows against torch.log_softmax in float64 (a library
    routine) at temperature 1 and tau."""
    import torch
    rng = np.random.default_rng(17)
    x = rng.normal(scale=3.0, size=(16, V)).astype(np.float32)
    tok = rng.integers(0, V, 16).astype(np.int32)
    for tau in (0.25, 0.6):
        lp0, lq = row_logprobs(x, "f32", V, tok, tau)
        t = torch.from_numpy(x.astype(np.float64))
        i = torch.arange(16)
        j = torch.from_numpy(tok).long()
        np.testing.assert_allclose(lp0, torch.log_softmax(t, 1)[i, j].numpy(), rtol=1e-12)
        np.testing.assert_allclose(lq, torch.log_softmax(t / tau, 1)[i, j].numpy(), rtol=1e-12)


def pin_dominant_token(row_logprobs, V=1000):
    """One logit 30 above the rest: lq = -log1p((V-1) e^(-30/tau)) ~ -1e-50 must
    keep its relative accuracy (a log of the full sum would round it to 0)."""
    x = np.zeros((1, V), dtype=np.float32)
    x[0, 5] = 30.0
    lp0, lq = row_logprobs(x, "f32", V, np.array([5], np.int32), 0.25)
    np.testing.assert_allclose(lq[0], -math.log1p((V - 1) * math.exp(-120.0)), rtol=1e-10)
    np.testing.assert_allclose(lp0[0], -math.log1p((V - 1) * math.exp(-30.0)), rtol=1e-10)


# ---- next rows: entropy, epsilon classes, carry-over, tree construction -----

def pin_entropy_library(entropy, V=700):
    """entropy(x float32 [n, V]) against torch.distributions.Categorical in
    float64 (a library routine), on rows with a peaked id and masked (-inf)
    entries: catches a dropped normaliser, a sign error or a wrong base."""
    import torch
    rng = np.random.default_rng(21)
    x = rng.normal(scale=3.0, size=(24, V)).astype(np.float32)
    x[:, 3] += 10.0
    x[5, 100:] = -np.inf
    want = torch.distributions.Categorical(logits=torch.from_numpy(x.astype(np.float64))).entropy()
    np.testing.assert_allclose(entropy(x), want.numpy(), rtol=1e-10, atol=1e-13)


def pin_entropy_uniform(entropy, V=1024):
    """Uniform rows have H = log V exactly (closed form)."""
    x = np.full((3, V), 1.25, np.float32)
    np.testing.assert_allclose(entropy(x), math.log(V), rtol=1e-12)


def pin_eps_classes(eps_class):
    """Constructed values on both sides of eps and 1 - eps (section 3.3):
    A <= eps is certain reject (0), A >= 1 - eps certain accept (2)."""
    A = np.array([1.0, 0.995, 0.99, 0.5, 0.0101, 0.0099, 0.001, 0.0, np.nan])
    with np.errstate(divide="ignore"):
        la = np.log(A)
    assert list(eps_class(la, 0.01)) == [2, 2, 2, 1, 1, 0, 0, 0, -1]


def pin_carry_example5(carry_state):
    """Example 5's walk reaches y = x_{0:c1} + y: the carried state takes the
    previous values up to the root's cut, root rows up to c1, then y's rows
    (rows are named by their index, so any misplaced position shows)."""
    T, c1, c2 = 16, 9, 4
    lay = assemble_layout([example5_tree(T, c1, c2)])
    rc = int(lay.seg_cut[0])
    prev = np.full((1, T), -7.0)
    vals = np.arange(lay.n_rows, dtype=np.float64) + 0.5
    out = carry_state(lay, np.array([1]), {"lp0": vals}, {"lp0": prev})
    want = np.empty(T)
    for t in range(1, T + 1):
        if t <= rc:
            want[t - 1] = -7.0
        elif t <= c1:
            want[t - 1] = lay.seg_row0[0] + (t - rc - 1) + 0.5
        else:
            want[t - 1] = lay.seg_row0[1] + (t - c1 - 1) + 0.5
    assert np.array_equal(out["lp0"][0], want)


def pin_bfs_example2(bfs):
    """The pages' Example 2 (golden fixture): the first expansion's cut is
    feasible under the root, its acceptance child expands next, the rejection
    child keeps the root's cut."""
    with open(os.path.join(GOLDEN, "example2_bfs.json")) as fh:
        g = json.load(fh)
    T, c1, c2 = 20, 11, 6
    t = bfs(T, g["n_pf"], None, [c1, c2])
    assert t["acc"][0] == 1 and t["acc"][1] == 3 and t["rej"][0] == 2
    assert list(t["seg_cut"][1:]) == [c1, c2] and list(t["seg_src"][1:]) == [0, 1]
    assert t["req"][0] == 1 and t["req"][1] == 2 and t["node_cut"][0] == T


def pin_bfs_condition1(bfs, trials=300):
    """Condition 1 on random BFS trees: every scored request's cut is <= its
    node's cut and its from-state's cut; deferred requests are the infeasible
    ones; rejection children keep their parent's cut."""
    rng = np.random.default_rng(1)
    for _ in range(trials):
        T = int(rng.integers(1, 50))
        cuts = rng.integers(0, T, 200)
        t = bfs(T, int(rng.integers(0, 15)), None if rng.random() < .5 else 4, cuts)
        for v, r in enumerate(t["req"]):
            if r >= 0:
                assert t["seg_cut"][r] <= t["node_cut"][v]
                src = t["seg_src"][r]
                assert t["seg_cut"][r] <= (T if src == 0 else t["seg_cut"][src])
            elif r == -2:
                assert t["deferred"][v] > t["node_cut"][v]
        for v in range(len(t["acc"])):
            if t["rej"][v] >= 0:
                assert t["node_cut"][t["rej"][v]] == t["node_cut"][v]


def pin_dp_brute_force(allocation_dp, allocation_brute, reaching_weights, trials=40):
    """eq. (19) against exhaustive search over ancestor-closed selections
    (Proposition 2), and Lemma 1: the value is the selection's reaching weight."""
    rng = np.random.default_rng(2)
    for _ in range(trials):
        acc, rej = [-1], [-1]
        frontier = [(0, 0)]
        while frontier:
            v, d = frontier.pop()
            if d < 3 and rng.random() < 0.85:
                a, b = len(acc), len(acc) + 1
                acc += [-1, -1]
                rej += [-1, -1]
                acc[v], rej[v] = a, b
                frontier += [(a, d + 1), (b, d + 1)]
        n = len(acc)
        acc, rej = np.array(acc), np.array(rej)
        cand = rng.random(n) < 0.8
        cand[0] = True
        h = rng.uniform(0.02, 0.98, n)
        for budget in range(0, 6):
            v, sel = allocation_dp(acc, rej, cand, h, budget)
            assert abs(v - allocation_brute(acc, rej, cand, h, budget)) <= 1e-12
            R = reaching_weights(acc, rej, h)
            assert sel.sum() <= budget and abs(R[sel].sum() - v) <= 1e-12
