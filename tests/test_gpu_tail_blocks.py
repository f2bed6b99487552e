"""The scoring kernel's tail blocks.

On a batch where every warp streams at least 2048 chunks, the last 1/16 of
the chunks is cut into small blocks that the warps finishing their own range
first take at run time.  A row that runs through several ranges (a warp's
range and tail blocks, or several tail blocks) is merged from one partial per
range in range order, so the per-row values of PreSTO eq. (6) (log p0 and
log q_tau of each token, Appendix B.1) must not depend on which warp took
which block.  Tail blocks are taken by the scoring kernel without entropy:
the full-size parity tests compare every row of its runs with the oracle
(configurations 3, 4 and the sweep points all have tail blocks there); these
tests check the order independence and the no-allocation entry point, whose
smaller static array gives it fewer, larger blocks.
"""

import numpy as np
import pytest
import torch

import mh_prefetch_subtree_gb300 as ps
from synth import make_workload
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def w4():
    # configuration 4: 45,820 rows of 128 chunks (V = 262,144 bf16)
    w = make_workload(4, device=DEV)
    warps = torch.cuda.get_device_properties(0).multi_processor_count * 16
    assert w.n_rows * 128 >= 2048 * warps, "the batch is too small to have tail blocks"
    yield w
    del w
    torch.cuda.empty_cache()


def test_tail_blocks_do_not_depend_on_the_order(w4):
    # three rounds of the scoring kernel without entropy (the one with tail
    # blocks) take the blocks in different orders; the bits stay the same
    runs = [H.run_gpu(w4, entropy=False) for _ in range(3)]
    assert runs[0]["status"] == 0 and runs[0]["wstatus"] == 0
    assert runs[0].get("entropy") is None
    for k in ("lp0", "lq", "log_accept", "state_seg", "path"):
        for r in runs[1:]:
            assert np.array_equal(runs[0][k], r[k], equal_nan=True), k


def test_tail_blocks_in_the_static_array_of_the_no_alloc_entry_point(w4):
    # the no-allocation entry point's blocks are larger; its per-row values
    # agree with the workspace path's within the per-token tolerance and its
    # log A within the log A tolerance
    w = w4
    ref = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                  V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    ref.score()
    torch.cuda.synchronize()
    assert int(ref.t["status"].item()) == 0
    f64 = lambda n: torch.full((n,), float("nan"), dtype=torch.float64, device=DEV)
    t = dict(lp0=f64(w.n_rows), lq=f64(w.n_rows), log_accept=f64(w.layout.n_seg),
             status=torch.zeros(1, dtype=torch.int32, device=DEV))
    ps.ps_score_subtree_noalloc(ref.batch, ps.make_score_out(**t))
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0, ps.dev_status_names(int(t["status"].item()))
    for k in ("lp0", "lq"):
        a, b = t[k].cpu().numpy(), ref.t[k].cpu().numpy()
        assert np.all(np.abs(a - b) <= H.TOK_RTOL * np.abs(b) + 1e-300), k
    req = ~w.layout.is_root()
    la, lb = t["log_accept"].cpu().numpy()[req], ref.t["log_accept"].cpu().numpy()[req]
    assert np.all(np.abs(la - lb) <= H.LA_ATOL)


def test_tail_blocks_with_float32_rows_match_the_oracle():
    # float32 rows of V = 151,936 (149 chunks, the last one ragged), 43,663 rows
    # (26.5 GB): every row of both scoring kernels against the oracle
    from synth.trees import assemble_layout, bfs_tree
    from synth.workload import Workload, draw_tokens, gen_logits
    rng = np.random.default_rng(74)
    lay = assemble_layout([bfs_tree(rng, 256, 8) for _ in range(30)])
    warps = torch.cuda.get_device_properties(0).multi_processor_count * 16
    assert lay.n_rows * 149 >= 2048 * warps, "the batch is too small to have tail blocks"
    x = gen_logits("boosted", dict(sigma=3.0, margin_mean=4.0), lay.n_rows, 151936, "f32",
                   seed=75, device=DEV)
    tok = draw_tokens(x, 0.25, seed=76)
    w = Workload(name="f32 tail blocks", layout=lay, V=151936, dtype="f32", alpha=4.0, tau=0.25,
                 logits=x, tokens=tok, u=1.0 - rng.random(lay.n_seg), max_steps=100)
    s = H.full_parity(w)
    assert s["lp0_max_rel_no_entropy"] <= H.TOK_RTOL
    del w, x, tok
    torch.cuda.empty_cache()


def test_tail_blocks_at_a_general_temperature(w4):
    # tau = 0.3 (1/tau not a power of two: a second exponential per logit), no
    # entropy: every row that reaches into the tail region and 2,000 others
    # against the oracle
    import oracle
    from oracle.hostcopy import bf16_bits
    w = w4
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=0.3, max_steps=w.max_steps)
    d.score_rows()
    torch.cuda.synchronize()
    assert int(d.t["status"].item()) == 0, ps.dev_status_names(int(d.t["status"].item()))
    n = w.n_rows
    tail0 = n - n // 16 - 1
    rng = np.random.default_rng(6)
    sel = np.unique(np.concatenate([np.arange(tail0, n), rng.choice(tail0, 2000, replace=False)]))
    idx = torch.from_numpy(sel).to(DEV)
    o = oracle.row_logprobs(bf16_bits(w.logits[idx]), "bf16", w.V, w.tokens[idx].cpu().numpy(),
                            0.3, entropy=False)
    g = {"lp0": d.t["lp0"].cpu().numpy()[sel], "lq": d.t["lq"].cpu().numpy()[sel]}
    H.check_rows(g, {"lp0": o[0], "lq": o[1]})
    del d
    torch.cuda.empty_cache()
