"""Pins for the oracle's round carry-over (section 3.2 step (3): the sampler
keeps the reached state's token-level log-probabilities) and for suffix sums
whose current-state values are carried instead of scored."""

import math

import numpy as np

import oracle
from synth.trees import assemble_layout, bfs_tree, example5_tree


def _ids(layout):
    """Per-row values that name the row: row r -> r + 0.5."""
    return np.arange(layout.n_rows, dtype=np.float64) + 0.5


def test_example5_reached_state_is_y():
    T, c1, c2 = 16, 9, 4
    lay = assemble_layout([example5_tree(T, c1, c2)])
    rc = int(lay.seg_cut[0])
    prev = np.full((1, T), -7.0)
    vals = _ids(lay)
    out = oracle.carry_state(lay, np.array([1]), {"lp0": vals}, {"lp0": prev})
    want = np.empty(T)
    for t in range(1, T + 1):
        if t <= rc:
            want[t - 1] = -7.0                                   # carried
        elif t <= c1:
            want[t - 1] = lay.seg_row0[0] + (t - rc - 1) + 0.5  # root rows
        else:
            want[t - 1] = lay.seg_row0[1] + (t - c1 - 1) + 0.5  # y's rows
    assert np.array_equal(out["lp0"][0], want)


def test_rejections_keep_the_current_state():
    rng = np.random.default_rng(1)
    lay = assemble_layout([bfs_tree(rng, 20, 6)])
    T = lay.T
    rc = int(lay.seg_cut[0])
    prev = np.arange(T, dtype=np.float64)[None, :] - 100.0
    vals = _ids(lay)
    out = oracle.carry_state(lay, np.array([0]), {"lp0": vals}, {"lp0": prev})
    assert np.array_equal(out["lp0"][0, :rc], prev[0, :rc])
    assert np.array_equal(out["lp0"][0, rc:], vals[lay.seg_row0[0]:lay.seg_row0[1]])


def test_loglik_and_confidence_closed_form():
    # uniform rows everywhere: every lp0 = -log V and every entropy = log V
    rng = np.random.default_rng(2)
    lay = assemble_layout([bfs_tree(rng, 12, 4), bfs_tree(rng, 12, 3)])
    V = 77
    T = lay.T
    x = np.full((lay.n_rows, V), 0.25, np.float32)
    tok = rng.integers(0, V, lay.n_rows).astype(np.int32)
    lp0, lq, ent = oracle.row_logprobs(x, "f32", V, tok, 0.25, entropy=True)
    prev = {k: np.full((2, T), v) for k, v in (("lp0", -math.log(V)), ("lq", -math.log(V)),
                                                 ("entropy", math.log(V)))}
    for state in (np.array([0, int(lay.chain_seg0[1])]), np.array([1, int(lay.chain_seg0[1]) + 1])):
        out = oracle.carry_state(lay, state, {"lp0": lp0, "lq": lq, "entropy": ent}, prev)
        np.testing.assert_allclose(out["loglik"], -math.log(V), rtol=1e-13)
        np.testing.assert_allclose(out["confidence"], -math.log(V), rtol=1e-13)


def test_carried_root_gives_the_same_sums_as_scored_root_rows():
    # two MH rounds: the second round's current state is the first round's reached state, given
    # once as scored rows and once as carried per-position values
    rng = np.random.default_rng(3)
    T, V = 24, 60
    for trial in range(20):
        lay1 = assemble_layout([bfs_tree(rng, T, 5)])
        x1 = rng.normal(scale=2.0, size=(lay1.n_rows, V)).astype(np.float32)
        t1 = rng.integers(0, V, lay1.n_rows).astype(np.int32)
        lp0_1, lq_1 = oracle.row_logprobs(x1, "f32", V, t1, 0.25)
        sums1 = oracle.suffix_sums(lay1, lp0_1, lq_1)
        _, la1 = oracle.log_accept(sums1, 4.0)
        u1 = 1.0 - rng.random(lay1.n_seg)
        wk = oracle.walk(lay1, la1, u1, 100)
        # the first round's root covers positions rc+1..T; its prefix is carried from
        # an earlier round (arbitrary values here)
        rc1 = int(lay1.seg_cut[0])
        prev = {"lp0": rng.normal(size=(1, T)), "lq": rng.normal(size=(1, T))}
        carried = oracle.carry_state(lay1, wk["state_seg"], {"lp0": lp0_1, "lq": lq_1}, prev)

        # the second round's tree, with the root's positions carried (root cut = T: no rows)
        tree2 = bfs_tree(rng, T, 4)
        tree2.finalize_root_cut(T)
        lay2c = assemble_layout([tree2])
        n_req_rows = lay2c.n_rows
        x2 = rng.normal(scale=2.0, size=(n_req_rows, V)).astype(np.float32)
        t2 = rng.integers(0, V, n_req_rows).astype(np.int32)
        lp0_2, lq_2 = oracle.row_logprobs(x2, "f32", V, t2, 0.25)
        sc = oracle.suffix_sums(lay2c, lp0_2, lq_2, root_lp0=carried["lp0"],
                               root_lq=carried["lq"])

        # the same second round with the root given as rows: rows for positions
        # 1..T whose values are the carried ones
        tree2.finalize_root_cut(0)
        lay2r = assemble_layout([tree2])
        lp0_r = np.concatenate([carried["lp0"][0], lp0_2])
        lq_r = np.concatenate([carried["lq"][0], lq_2])
        sr = oracle.suffix_sums(lay2r, lp0_r, lq_r)
        for k in ("lp_y", "lq_y", "lp_x", "lq_x"):
            assert np.array_equal(sc[k], sr[k], equal_nan=True), (trial, k)
        del rc1
