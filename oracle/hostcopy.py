"""Host copies of device-resident inputs, in the form the oracle reads.

TEST INFRASTRUCTURE, like the rest of this package: only the tests, the
package's ``smoke()`` check and the CPU-baseline legs of ``bench.py`` use it.
Nothing here computes the method: it moves logits rows from wherever torch
keeps them to host numpy arrays (bf16 as raw uint16 bit patterns, float32 as
is) and hands them, block by block, to ``oracle.row_logprobs``.
"""

from __future__ import annotations

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of the same bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def logits_np(t: torch.Tensor) -> tuple[np.ndarray, str]:
    """Host copy of a logits tensor and its dtype name ("bf16" or "f32")."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t), "bf16"
    assert t.dtype == torch.float32
    return t.detach().cpu().contiguous().numpy(), "f32"


def oracle_rows(w, block_rows: int = 8192, threads: int | None = None, entropy: bool = True,
                n_rows: int | None = None, rows: np.ndarray | None = None):
    """The oracle's per-row values (lp0, lq, entropy) of a workload ``w``
    (``synth.Workload``), copying its logits to the host block by block.

    entropy=False skips the entropy (returned as NaN).  n_rows limits the rows
    scored to the first n_rows; ``rows`` (sorted scored-row ids) limits them to
    a sample.  With a row index, each distinct (logits row, token) pair is
    scored once and the values are spread back to the rows that use it.
    """
    import oracle
    if rows is not None:
        sel = np.asarray(rows, dtype=np.int64)
    else:
        sel = np.arange(w.n_rows if n_rows is None else min(n_rows, w.n_rows), dtype=np.int64)
    toks = w.tokens.cpu().numpy()[sel]
    if w.row_index is not None:
        src = w.row_index.cpu().numpy()[sel].astype(np.int64)
    else:
        src = sel
    key = src * (w.V + 1) + toks
    uk, inv = np.unique(key, return_inverse=True)
    src_rows = (uk // (w.V + 1)).astype(np.int64)
    src_tok = (uk % (w.V + 1)).astype(np.int32)
    a0 = np.empty(uk.shape[0])
    aq = np.empty(uk.shape[0])
    ae = np.full(uk.shape[0], np.nan)
    for i0 in range(0, uk.shape[0], block_rows):
        i1 = min(uk.shape[0], i0 + block_rows)
        r = src_rows[i0:i1]
        if r[-1] - r[0] == i1 - i0 - 1:            # a contiguous block: a plain slice
            host = w.logits[int(r[0]):int(r[-1]) + 1]
        else:
            host = w.logits.index_select(0, torch.from_numpy(r).to(w.logits.device))
        lg, dt = logits_np(host)
        res = oracle.row_logprobs(lg, dt, w.V, src_tok[i0:i1], w.tau, threads=threads,
                                  entropy=entropy)
        a0[i0:i1], aq[i0:i1] = res[0], res[1]
        if entropy:
            ae[i0:i1] = res[2]
    return a0[inv], aq[inv], ae[inv]
