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
    mid = (E2M1_MAGNITUDES[1:] + E2M1_MAGNITUDES[:-1]) / 2      # 0.25, 0.75, ..., 5
    code = np.searchsorted(mid, a, side="left")                    # midpoints strictly below a
    tie = (code < mid.size) & (a == mid[np.minimum(code, mid.size - 1)])
    code = np.where(tie & (code % 2 == 1), code + 1, code).astype(np.uint8)  # a tie goes to the even code
    sign = (np.signbit(x) & (code != 0)).astype(np.uint8) << 3
    return code | sign


def pack_e2m1(codes) -> np.ndarray:
    """[rows, K] E2M1 codes -> [rows, K / 2] bytes, element 2t in the low four bits."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def mx_quantize(x, block: int = 32, rows_per_chunk: int = 512):
    """[rows, K] floats -> (packed E2M1 codes [rows, K / 2], E8M0 scale codes [rows, K / block])."""
    x = np.asarray(x)
    rows, K = x.shape
    packed = np.empty((rows, K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // block), dtype=np.uint8)
    for r0 in range(0, rows, rows_per_chunk):
        blocks = x[r0:r0 + rows_per_chunk].astype(np.float64).reshape(-1, K // block, block)
        amax = np.abs(blocks).max(axis=-1)
        X = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, -127)
        X = np.clip(X, -127, 127)
        codes = to_e2m1_codes(blocks / np.exp2(X)[..., None]).reshape(-1, K)
        packed[r0:r0 + rows_per_chunk] = pack_e2m1(codes)
        scales[r0:r0 + rows_per_chunk] = (X + 127).astype(np.uint8)
    return packed, scales
