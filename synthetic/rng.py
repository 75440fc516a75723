"""Counter-based SplitMix64 draws (uniform, normal, small integers) in numpy.

Large draws are split into chunks evaluated on a thread pool; numpy releases
the GIL inside its ufuncs, and each value depends only on its index, so the
result is identical for any chunking.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

STREAM_A = 0
STREAM_B = 1
STREAM_SA = 2
STREAM_SB = 3

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z):
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([seed], dtype=np.uint64) * _GOLDEN + np.uint64(stream + 1)
    return _mix64(z)[0]


def _raw(key: np.uint64, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * _GOLDEN)


def splitmix64_stream(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs x(start) .. x(start + count - 1)."""
    return _raw(_key(seed, stream), start, count)


def _chunked(total: int, fn, out: np.ndarray):
    spans = [(s, min(total, s + _CHUNK)) for s in range(0, total, _CHUNK)]
    if len(spans) <= 1:
        for s, e in spans:
            out[s:e] = fn(s, e - s)
        return out
    workers = min(len(spans), os.cpu_count() or 1, 16)

    def run(span):
        s, e = span
        out[s:e] = fn(s, e - s)

    with ThreadPoolExecutor(max_workers=workers) as pool:
        list(pool.map(run, spans))
    return out


def uniform(seed: int, stream: int, shape, lo: float, hi: float) -> np.ndarray:
    """float64 draws, uniform on [lo, hi)."""
    total = int(np.prod(shape))
    key = _key(seed, stream)
    scale = np.float64(2.0 ** -53)

    def fn(s, c):
        u = (_raw(key, s, c) >> np.uint64(11)).astype(np.float64) * scale
        return lo + (hi - lo) * u

    return _chunked(total, fn, np.empty(total, dtype=np.float64)).reshape(shape)


def normal(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """float64 draws, N(mean, std^2), one Box-Muller pair per value."""
    total = int(np.prod(shape))
    key = _key(seed, stream)
    scale = np.float64(2.0 ** -53)

    def fn(s, c):
        x = _raw(key, 2 * s, 2 * c)
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * scale
        return mean + std * (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2))

    return _chunked(total, fn, np.empty(total, dtype=np.float64)).reshape(shape)


def integers(seed: int, stream: int, shape, lo: int, hi: int) -> np.ndarray:
    """float64 draws of integers uniform on [lo, hi] (inclusive)."""
    total = int(np.prod(shape))
    key = _key(seed, stream)
    scale = np.float64(2.0 ** -53)
    span = float(hi - lo + 1)

    def fn(s, c):
        u = (_raw(key, s, c) >> np.uint64(11)).astype(np.float64) * scale
        return np.floor(u * span) + lo

    return _chunked(total, fn, np.empty(total, dtype=np.float64)).reshape(shape)
