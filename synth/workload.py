"""Seeded synthetic workloads shaped like the five benchmark configurations.

The pages measure on real LLMs and datasets that are not available here, so
these seeded stand-ins supply rows of logits with the stated vocabulary sizes
and value distributions, prefetching trees built by the pages' traversal rules,
proposal tokens drawn from the proposal law q_tau of each row (Gumbel-max on
logits / tau, i.e. the law of eq. (5)), and acceptance uniforms.

Logits are generated with a seeded ``torch.Generator`` on the requested device
(normally the GPU, because the larger configurations hold 3-31 GB of logits);
the same bytes are then given to both the CUDA path and the oracle.
Trees, cuts and uniforms come from numpy's PCG64 and are identical on every
machine.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from .trees import Layout, assemble_layout, bfs_tree, draw_uniforms, spine_tree

BASE_SEED = 10086   # the pages' seed (Table 6); config k uses BASE_SEED + k

CONFIGS = {
    1: dict(name="tiny-oracle V=1024 f32 T=64 Npf=8 depth4",
            V=1024, dtype="f32", T=64, n_pf=8, depth_cap=4, max_steps=4,
            alpha=4.0, tau=0.25, tree="bfs", n_chains=1,
            logits=("normal", dict(sigma=2.0))),
    2: dict(name="qwen3-vocab V=151936 bf16 T=1024 Npf=16",
            V=151936, dtype="bf16", T=1024, n_pf=16, depth_cap=None, max_steps=100,
            alpha=4.0, tau=0.25, tree="bfs", n_chains=1,
            logits=("boosted", dict(sigma=3.0, margin_mean=4.0))),
    3: dict(name="long-context V=151936 bf16 T=3072 Npf=64 spine30",
            V=151936, dtype="bf16", T=3072, n_pf=64, depth_cap=None, max_steps=100,
            alpha=4.0, tau=0.25, tree="spine", spine_depth=30, p_rej=0.97,
            target_tokens=100_000, n_chains=1,
            logits=("boosted", dict(sigma=3.0, margin_mean=4.0))),
    4: dict(name="gemma-vocab V=262144 bf16 T=2048 Npf=32 peaked",
            V=262144, dtype="bf16", T=2048, n_pf=32, depth_cap=None, max_steps=100,
            alpha=4.0, tau=0.25, tree="bfs", n_chains=1,
            logits=("dominant", dict(sigma=4.5, margin_mu=8.0, margin_sd=2.0))),
}

# config 5: 256 independent chains per sweep point over these grids
SWEEP5 = dict(n_chains=256, n_pf=(4, 8, 16, 32), T=(512, 1024, 2048),
              alpha=(2.0, 4.0, 8.0), V=151936, dtype="bf16",
              logits=("boosted", dict(sigma=3.0, margin_mean=4.0)))


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gen_logits(kind: str, params: dict, n_rows: int, V: int, dtype: str,
               seed: int, device="cpu", chunk_rows: int = 2048,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """Rows of synthetic logits, generated chunk by chunk.

    kind = "normal":   l_j ~ N(0, sigma^2)
    kind = "boosted":  N(0, sigma^2), then one uniformly chosen id per row is set
                       to (max of the other logits) + margin, margin ~ Exp(mean)
    kind = "dominant": N(0, sigma^2), then one uniformly chosen id per row is set
                       to (max of the other logits) + margin, margin ~ N(mu, sd^2)
    """
    g = _gen(seed, device)
    td = torch_dtype(dtype)
    if out is None:
        out = torch.empty((n_rows, V), dtype=td, device=device)
    sigma = float(params["sigma"])
    for r0 in range(0, n_rows, chunk_rows):
        r1 = min(n_rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0, V), generator=g, device=device, dtype=torch.float32)
        x.mul_(sigma)
        if kind != "normal":
            n = r1 - r0
            ids = torch.randint(0, V, (n,), generator=g, device=device)
            ar = torch.arange(n, device=device)
            x[ar, ids] = float("-inf")
            mx = x.max(dim=1).values
            if kind == "boosted":
                e = torch.empty(n, device=device).exponential_(
                    1.0 / float(params["margin_mean"]), generator=g)
            elif kind == "dominant":
                e = torch.randn(n, generator=g, device=device) * float(params["margin_sd"])
                e += float(params["margin_mu"])
            else:
                raise ValueError(kind)
            x[ar, ids] = mx + e
        out[r0:r1].copy_(x.to(td))
        del x
    return out


def draw_tokens(logits: torch.Tensor, tau: float, seed: int,
                chunk_rows: int = 2048, V: int | None = None) -> torch.Tensor:
    """One token per row drawn from softmax(logits / tau) by Gumbel-max.

    This stands in for the proposal LLM sampling y_t ~ q_tau (eq. (5)).
    """
    dev = logits.device
    g = _gen(seed, dev)
    n = logits.shape[0]
    V = logits.shape[1] if V is None else V
    tok = torch.empty(n, dtype=torch.int32, device=dev)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        u = torch.rand((r1 - r0, V), generator=g, device=dev, dtype=torch.float32)
        u.clamp_(min=1e-30)
        gumbel = u.log_().neg_().log_().neg_()
        z = logits[r0:r1, :V].float().div_(float(tau)).add_(gumbel)
        tok[r0:r1] = z.argmax(dim=1).to(torch.int32)
        del u, gumbel, z
    return tok


@dataclass
class Workload:
    """One subtree batch: layout, logits, tokens, uniforms and parameters."""

    name: str
    layout: Layout
    V: int
    dtype: str
    alpha: float
    tau: float
    logits: torch.Tensor          # [n_logit_rows, ld] in dtype
    tokens: torch.Tensor          # int32 [n_rows]
    u: np.ndarray                 # float64 [n_seg] acceptance uniforms (roots unused)
    max_steps: int
    row_index: torch.Tensor | None = None   # int64 [n_rows] or None (identity)
    info: dict = field(default_factory=dict)

    @property
    def ld(self) -> int:
        return int(self.logits.shape[1])

    @property
    def n_rows(self) -> int:
        return self.layout.n_rows

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logits_bytes(self) -> int:
        """Bytes of logits one scoring pass reads (rows x V x element size)."""
        return self.n_rows * self.V * self.elem_bytes


def _trees_for(cfg: dict, rng: np.random.Generator):
    if cfg["tree"] == "bfs":
        return [bfs_tree(rng, cfg["T"], cfg["n_pf"], cfg.get("depth_cap"))
                for _ in range(cfg.get("n_chains", 1))]
    if cfg["tree"] == "spine":
        # redraw (deterministically) until the scored suffix-token count is
        # within 10% of the target
        target = cfg["target_tokens"]
        for _attempt in range(10_000):
            t = spine_tree(rng, cfg["T"], cfg["n_pf"], cfg["spine_depth"],
                           cfg["p_rej"])
            if abs(t.suffix_tokens() - target) <= 0.1 * target:
                return [t]
        raise RuntimeError("spine tree target not reached")
    raise ValueError(cfg["tree"])


def make_workload(k: int, device="cpu", **override) -> Workload:
    """Build configuration k (1..4); keyword overrides shrink it for tests."""
    cfg = dict(CONFIGS[k])
    cfg.update(override)
    seed = int(cfg.get("seed", BASE_SEED + k))
    rng = np.random.default_rng(seed)
    trees = _trees_for(cfg, rng)
    layout = assemble_layout(trees)
    u = draw_uniforms(rng, layout.n_seg)
    kind, params = cfg["logits"]
    logits = gen_logits(kind, params, layout.n_rows, cfg["V"], cfg["dtype"],
                        seed=seed * 7 + 1, device=device)
    tokens = draw_tokens(logits, cfg["tau"], seed=seed * 7 + 2)
    return Workload(name=cfg["name"], layout=layout, V=cfg["V"], dtype=cfg["dtype"],
                    alpha=float(cfg["alpha"]), tau=float(cfg["tau"]), logits=logits,
                    tokens=tokens, u=u, max_steps=int(cfg["max_steps"]),
                    info=dict(config=k, seed=seed,
                              suffix_tokens=layout.suffix_tokens(),
                              n_requests=layout.n_seg - layout.n_chains))


SWEEP5_POOL_MIN_BYTES = 16 * 10**9     # distinct rows the sweep reads through its row index
SWEEP5_POOL_L2_MULT = 128              # and at least this many times the L2 cache


def sweep_pool_rows(V: int, elem_bytes: int, l2_bytes: int,
                    min_bytes: int = SWEEP5_POOL_MIN_BYTES) -> int:
    """Distinct logits rows in the pool of configuration 5: at least
    ``min_bytes`` and ``SWEEP5_POOL_L2_MULT`` x the L2 size, so that rows read in
    a shuffled order come from DRAM, not from the L2 cache."""
    row = -(-V * elem_bytes // 16) * 16
    need = max(int(min_bytes), SWEEP5_POOL_L2_MULT * int(l2_bytes))
    return -(-need // row)


def make_pool(n_pool: int, V: int, dtype: str, params: dict, taus, seed: int,
              device="cpu"):
    """A pool of distinct logits rows and one proposal token per (row, tau)."""
    logits = gen_logits("boosted", params, n_pool, V, dtype, seed=seed, device=device)
    toks = {float(t): draw_tokens(logits, float(t), seed=seed + 1 + i)
            for i, t in enumerate(taus)}
    return logits, toks


def workload_config5(pool_logits: torch.Tensor, pool_tokens: dict, n_pf: int, T: int,
                     alpha: float, n_chains: int = 256, seed: int | None = None,
                     V: int = SWEEP5["V"]) -> Workload:
    """One sweep point of configuration 5: independent BFS chains whose rows
    are read through a shuffled row index into a pool of distinct rows."""
    if seed is None:
        seed = BASE_SEED + 5 + 1000 * n_pf + T + int(alpha * 10)
    rng = np.random.default_rng(seed)
    trees = [bfs_tree(rng, T, n_pf) for _ in range(n_chains)]
    layout = assemble_layout(trees)
    u = draw_uniforms(rng, layout.n_seg)
    n_pool = pool_logits.shape[0]
    n = layout.n_rows
    reps = -(-n // n_pool)
    idx = np.concatenate([rng.permutation(n_pool) for _ in range(reps)])[:n]
    dev = pool_logits.device
    row_index = torch.from_numpy(idx.astype(np.int64)).to(dev)
    tau = 1.0 / alpha
    tokens = pool_tokens[float(tau)][row_index].to(torch.int32)
    dtype = "bf16" if pool_logits.dtype == torch.bfloat16 else "f32"
    return Workload(name=f"sweep chains={n_chains} Npf={n_pf} T={T} alpha={alpha}",
                    layout=layout, V=V, dtype=dtype, alpha=float(alpha), tau=tau,
                    logits=pool_logits, tokens=tokens, u=u, max_steps=100,
                    row_index=row_index,
                    info=dict(config=5, seed=seed, suffix_tokens=layout.suffix_tokens(),
                              n_requests=layout.n_seg - layout.n_chains, n_pool=n_pool))
