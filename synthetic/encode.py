"""Encode float draws as bf16 / E4M3 codes (input preparation only).

Draws are rounded to float32 first (round to nearest even), then cast with
torch's CPU conversions, which round to nearest even.  E4M3 values are
clamped to the finite range first (satfinite), so no draw becomes NaN.
"""
from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0


def to_bf16_codes(x) -> np.ndarray:
    """float array -> uint16 bf16 bit patterns (same shape)."""
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    t = torch.from_numpy(x32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_e4m3_codes(x) -> np.ndarray:
    """float array -> uint8 E4M3 (OCP E4M3FN) bit patterns, saturating."""
    x32 = np.clip(np.asarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(x32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()
