"""Small shared helpers for the tests (no scoring arithmetic)."""

from __future__ import annotations

import numpy as np
import torch


from oracle.hostcopy import bf16_bits, logits_np  # noqa: F401  (re-exported for the tests)


def bf16_from_float(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (uint16), via torch."""
    return bf16_bits(torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def float_from_bf16(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)
