"""Throughput metrics of a GEMM call (pure Python).

  flops  = 2 * M * N * K                       ("Gemm Optimization" guide, 8.1)
  bytes  = A + B + C + (M + N) * 4 for scaled 8-bit inputs   (same guide, 8.2)
  AI     = flops / bytes                       (same guide, 8.3)

M and N are the valid (unpadded) extents: padded-tile work is not counted.
"""
from __future__ import annotations


def gemm_flops(m: int, n: int, k: int) -> int:
    return 2 * m * n * k


def gemm_bytes(m: int, n: int, k: int, in_bytes: int = 2, out_bytes: int = 2, scaled: bool = False) -> int:
    b = m * k * in_bytes + n * k * in_bytes + m * n * out_bytes
    if scaled:
        b += (m + n) * 4
    return b


def arithmetic_intensity(m: int, n: int, k: int, in_bytes: int = 2, out_bytes: int = 2,
                         scaled: bool = False) -> float:
    return gemm_flops(m, n, k) / gemm_bytes(m, n, k, in_bytes, out_bytes, scaled)


def tflops(m: int, n: int, k: int, seconds: float) -> float:
    return gemm_flops(m, n, k) / seconds / 1e12


def gbps(nbytes: float, seconds: float) -> float:
    return nbytes / seconds / 1e9
