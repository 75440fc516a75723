"""Encode float draws as bf16 / E4M3 / MXFP4 codes (input preparation only).

Draws are rounded to float32 first (round to nearest even), then cast with
torch's CPU conversions, which round to nearest even.  E4M3 values are
clamped to the finite range first (satfinite), so no draw becomes NaN.

MXFP4 (OCP Microscaling, version 1.0, section 6.3 "Conversion"): each block of
32 consecutive values along a row shares the scale 2^X with
X = floor(log2(max |v|)) - 2 (2 being the largest exponent of E2M1), stored as
the E8M0 code X + 127; each value becomes the E2M1 code nearest v / 2^X
(ties to the even code, magnitudes above 6 saturate).  Codes are packed two to
a byte, element 2t in the low four bits of byte t.
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


E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # codes 0..7; bit 3 is the sign


def to_e2m1_codes(x) -> np.ndarray:
    """float array -> uint8 E2M1 codes (0..15), nearest, ties to even, saturating."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    dist = np.abs(a[..., None] - E2M1_MAGNITUDES)
    best = dist.min(axis=-1, keepdims=True)
    # among the nearest magnitudes take the even code (fraction bit 0)
    tie_ok = (dist == best) & ((np.arange(8) & 1) == 0)
    near = dist == best
    code = np.where(tie_ok.any(axis=-1), tie_ok.argmax(axis=-1), near.argmax(axis=-1)).astype(np.uint8)
    sign = (np.signbit(x) & (code != 0)).astype(np.uint8) << 3
    return code | sign


def pack_e2m1(codes) -> np.ndarray:
    """[rows, K] E2M1 codes -> [rows, K / 2] bytes, element 2t in the low four bits."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def mx_quantize(x, block: int = 32):
    """[rows, K] floats -> (packed E2M1 codes [rows, K / 2], E8M0 scale codes [rows, K / block])."""
    x = np.asarray(x, dtype=np.float64)
    rows, K = x.shape
    blocks = x.reshape(rows, K // block, block)
    amax = np.abs(blocks).max(axis=-1)
    with np.errstate(divide="ignore"):
        X = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, -127)
    X = np.clip(X, -127, 127)
    scaled = blocks / np.exp2(X)[..., None]
    codes = to_e2m1_codes(scaled).reshape(rows, K)
    return pack_e2m1(codes), (X + 127).astype(np.uint8)
