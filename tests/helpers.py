"""Small shared helpers for the tests (no scoring arithmetic)."""

from __future__ import annotations

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of the same bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def logits_np(t: torch.Tensor) -> tuple[np.ndarray, str]:
    """Host copy of a logits tensor in the form the oracle reads."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t), "bf16"
    assert t.dtype == torch.float32
    return t.detach().cpu().contiguous().numpy(), "f32"


def bf16_from_float(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (uint16), via torch."""
    return bf16_bits(torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def float_from_bf16(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)
