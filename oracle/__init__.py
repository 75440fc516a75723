"""Reference oracle for C = A . B^T (bf16 and E4M3 inputs, fp64 arithmetic),
for the linear layer around it (bias, GELU / SiLU, gated up projection), for
the block-scaled FP4 (MXFP4) product, and for E4M3 activations times E2M1
weights (W4A8).

TEST INFRASTRUCTURE ONLY.  The product library never imports this package;
only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use it.  It shares no code with the CUDA path: the arithmetic lives in
``gemm_oracle.c`` (plain C, fp64 triple loop, OpenMP over rows), compiled with
gcc by :func:`build` and loaded with ctypes.

Parity is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``
(identity and permutation products, rank-1 closed forms, all-ones, brute force
in exact rational arithmetic, decoder tables from the format definitions).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

BF16 = 0
E4M3 = 1

ACT_NONE = 0
ACT_GELU = 1
ACT_SILU = 2

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle into a shared library with gcc (-O2, OpenMP)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    c_i64 = ctypes.c_int64
    vp = ctypes.c_void_p
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = ctypes.c_double
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e4m3.restype = ctypes.c_double
    lib.oracle_round_bf16.argtypes = [ctypes.c_double]
    lib.oracle_round_bf16.restype = ctypes.c_uint16
    lib.oracle_round_bf16_n.argtypes = [vp, c_i64, vp]
    lib.oracle_round_bf16_n.restype = None
    lib.oracle_gemm.argtypes = [ctypes.c_int, vp, vp, vp, vp, c_i64, c_i64, c_i64, vp, vp]
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm_points.argtypes = [ctypes.c_int, vp, vp, vp, vp, c_i64, c_i64, c_i64,
                                       vp, vp, c_i64, vp, vp]
    lib.oracle_gemm_points.restype = ctypes.c_int
    lib.oracle_act.argtypes = [ctypes.c_int, ctypes.c_double]
    lib.oracle_act.restype = ctypes.c_double
    lib.oracle_linear.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, c_i64, c_i64, c_i64, ctypes.c_int,
                                  ctypes.c_int, vp, vp]
    lib.oracle_linear.restype = ctypes.c_int
    lib.oracle_linear_points.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, c_i64, c_i64, c_i64, ctypes.c_int,
                                         ctypes.c_int, vp, vp, c_i64, vp, vp]
    lib.oracle_linear_points.restype = ctypes.c_int
    lib.oracle_decode_e2m1.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e2m1.restype = ctypes.c_double
    lib.oracle_decode_e8m0.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e8m0.restype = ctypes.c_double
    lib.oracle_mxfp4_gemm.argtypes = [vp, vp, vp, vp, c_i64, c_i64, c_i64, vp, vp]
    lib.oracle_mxfp4_gemm.restype = ctypes.c_int
    lib.oracle_mxfp4_gemm_points.argtypes = [vp, vp, vp, vp, c_i64, c_i64, c_i64, vp, vp, c_i64, vp, vp]
    lib.oracle_mxfp4_gemm_points.restype = ctypes.c_int
    lib.oracle_w4a8_gemm.argtypes = [vp, vp, vp, vp, c_i64, c_i64, c_i64, vp, vp]
    lib.oracle_w4a8_gemm.restype = ctypes.c_int
    lib.oracle_w4a8_gemm_points.argtypes = [vp, vp, vp, vp, c_i64, c_i64, c_i64, vp, vp, c_i64, vp, vp]
    lib.oracle_w4a8_gemm_points.restype = ctypes.c_int
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _codes(x, dtype):
    want = np.uint16 if dtype == BF16 else np.uint8
    x = np.ascontiguousarray(x)
    if x.dtype != want:
        raise TypeError(f"expected {want} codes, got {x.dtype}")
    return x


def gemm(dtype, A, B, sa=None, sb=None, lib=None):
    """Full reference product.

    A: [m, K] codes (uint16 bf16 bits or uint8 E4M3 bits); B: [n, K] codes.
    sa [m], sb [n]: float32 scales (both or neither).
    Returns (C_ref, S_abs), both float64 [m, n].
    """
    lib = lib or load()
    A = _codes(A, dtype)
    B = _codes(B, dtype)
    m, K = A.shape
    n, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if (sa is None) != (sb is None):
        raise ValueError("give both scales or neither")
    if sa is not None:
        sa = np.ascontiguousarray(sa, dtype=np.float32)
        sb = np.ascontiguousarray(sb, dtype=np.float32)
        if sa.shape != (m,) or sb.shape != (n,):
            raise ValueError("scale lengths must be m and n")
    C = np.empty((m, n), dtype=np.float64)
    S = np.empty((m, n), dtype=np.float64)
    rc = lib.oracle_gemm(dtype, _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), m, n, K, _ptr(C), _ptr(S))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return C, S


def gemm_points(dtype, A, B, rows, cols, sa=None, sb=None, lib=None):
    """Reference values at the points (rows[p], cols[p]); returns (C_ref, S_abs)."""
    lib = lib or load()
    A = _codes(A, dtype)
    B = _codes(B, dtype)
    m, K = A.shape
    n, _ = B.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    if sa is not None:
        sa = np.ascontiguousarray(sa, dtype=np.float32)
        sb = np.ascontiguousarray(sb, dtype=np.float32)
    C = np.empty(rows.shape, dtype=np.float64)
    S = np.empty(rows.shape, dtype=np.float64)
    rc = lib.oracle_gemm_points(dtype, _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), m, n, K,
                                _ptr(rows), _ptr(cols), rows.size, _ptr(C), _ptr(S))
    if rc != 0:
        raise ValueError("oracle_gemm_points rejected its arguments")
    return C, S


def _linear_inputs(dtype, A, B, sa, sb, bias, gated):
    A = _codes(A, dtype)
    B = _codes(B, dtype)
    m, K = A.shape
    rows_b, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if gated and rows_b % 2:
        raise ValueError("a gated layer's B holds 2n rows")
    n = rows_b // 2 if gated else rows_b
    if (sa is None) != (sb is None):
        raise ValueError("give both scales or neither")
    if sa is not None:
        sa = np.ascontiguousarray(sa, dtype=np.float32)
        sb = np.ascontiguousarray(sb, dtype=np.float32)
        if sa.shape != (m,) or sb.shape != (rows_b,):
            raise ValueError("scale lengths must be m and the rows of B")
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        if bias.shape != (rows_b,):
            raise ValueError("bias length must be the rows of B")
    return A, B, sa, sb, bias, m, n, K


def linear(dtype, A, B, sa=None, sb=None, bias=None, act=ACT_NONE, gated=False, lib=None):
    """Reference linear layer: act(A . B^T (* scales) + bias), or with gated=True
    act(gate + b_gate) * (up + b_up) where B = [gate rows; up rows].
    Returns (Y_ref, E_abs), float64 [m, n]."""
    lib = lib or load()
    A, B, sa, sb, bias, m, n, K = _linear_inputs(dtype, A, B, sa, sb, bias, gated)
    Y = np.empty((m, n), dtype=np.float64)
    E = np.empty((m, n), dtype=np.float64)
    rc = lib.oracle_linear(dtype, _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), m, n, K, int(act),
                           int(bool(gated)), _ptr(Y), _ptr(E))
    if rc != 0:
        raise ValueError("oracle_linear rejected its arguments")
    return Y, E


def linear_points(dtype, A, B, rows, cols, sa=None, sb=None, bias=None, act=ACT_NONE, gated=False, lib=None):
    """Reference linear layer at the points (rows[p], cols[p]); returns (Y_ref, E_abs)."""
    lib = lib or load()
    A, B, sa, sb, bias, m, n, K = _linear_inputs(dtype, A, B, sa, sb, bias, gated)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    Y = np.empty(rows.shape, dtype=np.float64)
    E = np.empty(rows.shape, dtype=np.float64)
    rc = lib.oracle_linear_points(dtype, _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(bias), m, n, K, int(act),
                                  int(bool(gated)), _ptr(rows), _ptr(cols), rows.size, _ptr(Y), _ptr(E))
    if rc != 0:
        raise ValueError("oracle_linear_points rejected its arguments")
    return Y, E


def act(kind, x, lib=None):
    """The activation alone, elementwise over doubles."""
    lib = lib or load()
    x = np.asarray(x, dtype=np.float64)
    return np.array([lib.oracle_act(int(kind), float(v)) for v in x.ravel()]).reshape(x.shape)


def decode_bf16(bits, lib=None):
    lib = lib or load()
    bits = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.oracle_decode_bf16(int(b)) for b in bits.ravel()]).reshape(bits.shape)


def decode_e4m3(codes, lib=None):
    lib = lib or load()
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_decode_e4m3(int(c)) for c in codes.ravel()]).reshape(codes.shape)


def round_bf16(x, lib=None):
    """Round doubles to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_round_bf16_n(_ptr(x), x.size, _ptr(out))
    return out


def _mx_inputs(A, B, EA, EB):
    arrs = [np.ascontiguousarray(x) for x in (A, B, EA, EB)]
    for x in arrs:
        if x.dtype != np.uint8 or x.ndim != 2:
            raise TypeError("MXFP4 operands and scales are 2-D uint8 arrays")
    A, B, EA, EB = arrs
    m, half_k = A.shape
    n = B.shape[0]
    K = 2 * half_k
    if B.shape[1] != half_k or K % 32 != 0:
        raise ValueError("A and B hold K / 2 bytes per row, K a multiple of 32")
    if EA.shape != (m, K // 32) or EB.shape != (n, K // 32):
        raise ValueError("scales hold K / 32 bytes per row of A and of B")
    return A, B, EA, EB, m, n, K


def mxfp4_gemm(A, B, EA, EB, lib=None):
    """Full reference MXFP4 product.

    A [m, K/2], B [n, K/2]: packed E2M1 codes (element 2t in the low four bits
    of byte t); EA [m, K/32], EB [n, K/32]: E8M0 scale codes, one per block of
    32 elements along K.  Returns (C_ref, S_abs), float64 [m, n]."""
    lib = lib or load()
    A, B, EA, EB, m, n, K = _mx_inputs(A, B, EA, EB)
    C = np.empty((m, n), dtype=np.float64)
    S = np.empty((m, n), dtype=np.float64)
    if lib.oracle_mxfp4_gemm(_ptr(A), _ptr(B), _ptr(EA), _ptr(EB), m, n, K, _ptr(C), _ptr(S)) != 0:
        raise ValueError("oracle_mxfp4_gemm rejected its arguments")
    return C, S


def mxfp4_gemm_points(A, B, EA, EB, rows, cols, lib=None):
    """Reference MXFP4 values at the points (rows[p], cols[p]); returns (C_ref, S_abs)."""
    lib = lib or load()
    A, B, EA, EB, m, n, K = _mx_inputs(A, B, EA, EB)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    C = np.empty(rows.shape, dtype=np.float64)
    S = np.empty(rows.shape, dtype=np.float64)
    if lib.oracle_mxfp4_gemm_points(_ptr(A), _ptr(B), _ptr(EA), _ptr(EB), m, n, K, _ptr(rows), _ptr(cols),
                                    rows.size, _ptr(C), _ptr(S)) != 0:
        raise ValueError("oracle_mxfp4_gemm_points rejected its arguments")
    return C, S


def _w4a8_inputs(A, B, sa, sb):
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    if A.dtype != np.uint8 or B.dtype != np.uint8 or A.ndim != 2 or B.ndim != 2:
        raise TypeError("W4A8 operands are 2-D uint8 arrays")
    m, K = A.shape
    n = B.shape[0]
    if B.shape[1] * 2 != K:
        raise ValueError("B holds K / 2 bytes per row (two E2M1 codes a byte)")
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    if sa.shape != (m,) or sb.shape != (n,):
        raise ValueError("scale lengths must be m and n")
    return A, B, sa, sb, m, n, K


def w4a8_gemm(A, B, sa, sb, lib=None):
    """Full reference W4A8 product: A [m, K] E4M3 codes, B [n, K/2] packed E2M1
    codes (element 2t in the low four bits of byte t), sa [m], sb [n] fp32.
    Returns (C_ref, S_abs), float64 [m, n]."""
    lib = lib or load()
    A, B, sa, sb, m, n, K = _w4a8_inputs(A, B, sa, sb)
    C = np.empty((m, n), dtype=np.float64)
    S = np.empty((m, n), dtype=np.float64)
    if lib.oracle_w4a8_gemm(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), m, n, K, _ptr(C), _ptr(S)) != 0:
        raise ValueError("oracle_w4a8_gemm rejected its arguments")
    return C, S


def w4a8_gemm_points(A, B, sa, sb, rows, cols, lib=None):
    """Reference W4A8 values at the points (rows[p], cols[p]); returns (C_ref, S_abs)."""
    lib = lib or load()
    A, B, sa, sb, m, n, K = _w4a8_inputs(A, B, sa, sb)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    C = np.empty(rows.shape, dtype=np.float64)
    S = np.empty(rows.shape, dtype=np.float64)
    if lib.oracle_w4a8_gemm_points(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), m, n, K, _ptr(rows), _ptr(cols),
                                   rows.size, _ptr(C), _ptr(S)) != 0:
        raise ValueError("oracle_w4a8_gemm_points rejected its arguments")
    return C, S


def decode_e2m1(codes, lib=None):
    lib = lib or load()
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_decode_e2m1(int(c)) for c in codes.ravel()]).reshape(codes.shape)


def decode_e8m0(codes, lib=None):
    lib = lib or load()
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_decode_e8m0(int(c)) for c in codes.ravel()]).reshape(codes.shape)


def threads(lib=None) -> int:
    return (lib or load()).oracle_threads()
