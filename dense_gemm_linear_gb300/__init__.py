"""GB300 (sm_103a) dense linear-layer GEMM: C = A . B^T in bf16, E4M3 and MXFP4.

Python binding of the C ABI in ``include/dgl.h``.  Functions named ``dgl_*``
marshal plain integers/pointers into the library one to one; the ``gemm_*``
helpers take torch CUDA tensors, allocate the output with torch when none is
given, and call the same entry points on torch's current stream.  Every step
of the computation runs in the library's CUDA kernels; if the library is
missing, loading raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

from . import metrics  # noqa: F401  (pure-Python metric helpers)

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "_build", "libdgl.so")

DGL_OK = 0
DGL_ERR_ARG = -1
DGL_ERR_ALIGN = -2
DGL_ERR_SHAPE = -3
DGL_ERR_UNSUPPORTED = -4
DGL_ERR_CUDA = -5
DGL_ERR_TIMEOUT = -6

OUT_BF16 = 0
OUT_F32 = 1
DTYPE_BF16 = 0
DTYPE_E4M3 = 1
DTYPE_MXFP4 = 2
DTYPE_W4A8 = 3
PATH_TC = 0
PATH_DECODE = 1
PATH_EMPTY = 2
ACT_NONE = 0
ACT_GELU = 1
ACT_SILU = 2
K_MAJOR = 0
MN_MAJOR = 1

EXPORTED = ["dgl_gemm_bf16", "dgl_gemm_fp8", "dgl_gemm_planned", "dgl_plan", "dgl_tile_metrics",
            "dgl_device_status", "dgl_status_string", "dgl_version", "dgl_gemm_noalloc", "dgl_linear",
            "dgl_plan_linear", "dgl_gemm_bf16_ex", "dgl_gemm_mxfp4", "dgl_shutdown", "dgl_gemm_w4a8",
            "dgl_gemm_batch"]


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("tile_k", ctypes.c_int32), ("stages", ctypes.c_int32), ("cta_group", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("num_tiles", ctypes.c_int32), ("tile_eff", ctypes.c_double),
                ("wq_eff", ctypes.c_double), ("dim_eff", ctypes.c_double), ("est_us", ctypes.c_double),
                ("stream_k", ctypes.c_int32), ("split_tail", ctypes.c_int32), ("k_group", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class GemmDesc(ctypes.Structure):
    """One GEMM of dgl_gemm_batch (the C struct dgl_gemm_desc)."""
    _fields_ = [("dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("A", ctypes.c_void_p),
                ("B", ctypes.c_void_p), ("scale_a", ctypes.c_void_p), ("scale_b", ctypes.c_void_p),
                ("C", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("m_valid", ctypes.c_int64), ("n_valid", ctypes.c_int64)]


class DglError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lib = None


def load_library(path: str | None = None):
    """Load libdgl.so (build it first with ``_build.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with dense_gemm_linear_gb300._build.build()")
    lib = ctypes.CDLL(p)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.dgl_gemm_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
    lib.dgl_gemm_bf16.restype = i32
    lib.dgl_gemm_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
    lib.dgl_gemm_fp8.restype = i32
    lib.dgl_gemm_planned.argtypes = [i32, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32,
                                     ctypes.POINTER(PlanInfo), vp]
    lib.dgl_gemm_planned.restype = i32
    lib.dgl_gemm_noalloc.argtypes = [i32, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
    lib.dgl_gemm_noalloc.restype = i32
    lib.dgl_linear.argtypes = [i32, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, i32, i32,
                               ctypes.POINTER(PlanInfo), vp]
    lib.dgl_linear.restype = i32
    lib.dgl_plan_linear.argtypes = [i32, i64, i64, i64, i32, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.dgl_plan_linear.restype = i32
    lib.dgl_gemm_bf16_ex.argtypes = [i32, i32, vp, i64, vp, i64, vp, i64, i64, i64, i64, i32,
                                     ctypes.POINTER(PlanInfo), vp]
    lib.dgl_gemm_bf16_ex.restype = i32
    lib.dgl_gemm_w4a8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
    lib.dgl_gemm_w4a8.restype = i32
    lib.dgl_gemm_mxfp4.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
    lib.dgl_gemm_mxfp4.restype = i32
    lib.dgl_gemm_batch.argtypes = [ctypes.POINTER(GemmDesc), i32, vp]
    lib.dgl_gemm_batch.restype = i32
    lib.dgl_plan.argtypes = [i32, i64, i64, i64, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.dgl_plan.restype = i32
    lib.dgl_tile_metrics.argtypes = [i64, i64, i32, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.dgl_tile_metrics.restype = i32
    lib.dgl_shutdown.argtypes = []
    lib.dgl_shutdown.restype = i32
    lib.dgl_device_status.argtypes = [vp]
    lib.dgl_device_status.restype = i32
    lib.dgl_status_string.argtypes = [i32]
    lib.dgl_status_string.restype = ctypes.c_char_p
    lib.dgl_version.argtypes = []
    lib.dgl_version.restype = i32
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().dgl_status_string(status).decode()
    except ImportError:
        return "library not loaded"


def _check(status: int, where: str):
    if status != DGL_OK:
        raise DglError(status, where)


# ---------------------------------------------------------------- raw C-ABI calls
def dgl_gemm_bf16(A, B, C, M, N, K, m_valid=0, n_valid=0, out_dtype=OUT_BF16, stream=0) -> int:
    return load_library().dgl_gemm_bf16(A, B, C, M, N, K, m_valid, n_valid, out_dtype, stream)


def dgl_gemm_fp8(A, B, sa, sb, C, M, N, K, m_valid=0, n_valid=0, out_dtype=OUT_BF16, stream=0) -> int:
    return load_library().dgl_gemm_fp8(A, B, sa, sb, C, M, N, K, m_valid, n_valid, out_dtype, stream)


def gemm_descs(items):
    """A ctypes array of GemmDesc from dicts (or GemmDesc instances) for dgl_gemm_batch."""
    arr = (GemmDesc * len(items))()
    for i, it in enumerate(items):
        arr[i] = it if isinstance(it, GemmDesc) else GemmDesc(**it)
    return arr


def dgl_gemm_batch(items, stream=0) -> int:
    """Independent GEMMs back to back on one stream (see dgl_gemm_batch in dgl.h); items: GemmDesc array or list."""
    arr = items if isinstance(items, ctypes.Array) else gemm_descs(items)
    return load_library().dgl_gemm_batch(arr, len(arr), stream)


def dgl_gemm_mxfp4(A, B, sfa, sfb, C, M, N, K, m_valid=0, n_valid=0, out_dtype=OUT_BF16, stream=0) -> int:
    """Block-scaled FP4: A [m][K/2], B [n][K/2] packed E2M1 bytes; sfa [m][K/32], sfb [n][K/32] E8M0 bytes."""
    return load_library().dgl_gemm_mxfp4(A, B, sfa, sfb, C, M, N, K, m_valid, n_valid, out_dtype, stream)


def dgl_gemm_w4a8(A, B, sa, sb, C, M, N, K, m_valid=0, n_valid=0, out_dtype=OUT_BF16, stream=0) -> int:
    """E4M3 A [m][K] x packed E2M1 B [n][K/2] (two codes a byte), fp32 scales sa [m], sb [n]."""
    return load_library().dgl_gemm_w4a8(A, B, sa, sb, C, M, N, K, m_valid, n_valid, out_dtype, stream)


def dgl_gemm_planned(dtype, A, B, sa, sb, C, M, N, K, m_valid, n_valid, out_dtype, plan: PlanInfo,
                     stream=0) -> int:
    return load_library().dgl_gemm_planned(dtype, A, B, sa, sb, C, M, N, K, m_valid, n_valid, out_dtype,
                                           ctypes.byref(plan), stream)


def dgl_gemm_noalloc(dtype, A, B, sa, sb, C, M, N, K, m_valid=0, n_valid=0, out_dtype=OUT_BF16, stream=0) -> int:
    """The GEMM that allocates no device memory (stream-K partials in a fixed device array)."""
    return load_library().dgl_gemm_noalloc(dtype, A, B, sa, sb, C, M, N, K, m_valid, n_valid, out_dtype, stream)


def dgl_linear(dtype, A, B, sa, sb, bias, C, M, N, K, m_valid=0, n_valid=0, out_dtype=OUT_BF16, act=0, gated=0,
               plan: PlanInfo | None = None, stream=0) -> int:
    """Linear layer act(A . B^T + bias), or the gated form (see include/dgl.h)."""
    return load_library().dgl_linear(dtype, A, B, sa, sb, bias, C, M, N, K, m_valid, n_valid, out_dtype, act, gated,
                                     ctypes.byref(plan) if plan is not None else None, stream)


def dgl_gemm_bf16_ex(a_major, b_major, A, lda, B, ldb, C, ldc, m, n, K, out_dtype=OUT_BF16,
                     plan: PlanInfo | None = None, stream=0) -> int:
    """bf16 GEMM with K-major or MN-major operands and explicit pitches (see include/dgl.h)."""
    return load_library().dgl_gemm_bf16_ex(a_major, b_major, A, lda, B, ldb, C, ldc, m, n, K, out_dtype,
                                           ctypes.byref(plan) if plan is not None else None, stream)


def dgl_plan(dtype, m, n, K, out_dtype=OUT_BF16, num_sms=0) -> PlanInfo:
    info = PlanInfo()
    _check(load_library().dgl_plan(dtype, m, n, K, out_dtype, num_sms, ctypes.byref(info)), "dgl_plan")
    return info


def dgl_plan_linear(dtype, m, n, K, out_dtype=OUT_BF16, gated=0, num_sms=0) -> PlanInfo:
    info = PlanInfo()
    _check(load_library().dgl_plan_linear(dtype, m, n, K, out_dtype, int(gated), num_sms, ctypes.byref(info)),
           "dgl_plan_linear")
    return info


def dgl_tile_metrics(m, n, tile_m, tile_n, num_units) -> PlanInfo:
    info = PlanInfo()
    _check(load_library().dgl_tile_metrics(m, n, tile_m, tile_n, num_units, ctypes.byref(info)),
           "dgl_tile_metrics")
    return info


def dgl_device_status(stream=0) -> int:
    return load_library().dgl_device_status(stream)


def dgl_shutdown() -> int:
    """Free the library's workspaces and caches on the current device (see include/dgl.h)."""
    return load_library().dgl_shutdown()


def dgl_version() -> int:
    return load_library().dgl_version()


# ---------------------------------------------------------------- torch helpers
def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check_operand(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or t.stride(1) != 1 or t.stride(0) != t.shape[1]:
        raise ValueError(f"{name} must be a contiguous 2-D tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _out_tensor(out, m, n, out_dtype, device):
    import torch
    tdt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
    if out is None:
        return torch.empty((m, n), dtype=tdt, device=device), n, m
    if out.dtype != tdt or out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("out must be a 2-D row-major tensor of the output dtype")
    if out.shape[0] < m or out.stride(0) < n:
        raise ValueError("out is smaller than the valid region")
    return out, out.stride(0), out.shape[0]


def gemm_bf16(A, B, out=None, *, out_dtype=OUT_BF16, stream=None, plan: PlanInfo | None = None):
    """C = A . B^T for bf16 A [m, K], B [n, K] (CUDA tensors); returns C [m, n] (or `out`)."""
    import torch
    _check_operand(A, "A", torch.bfloat16)
    _check_operand(B, "B", torch.bfloat16)
    m, K = A.shape
    n, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    C, ldc, rows = _out_tensor(out, m, n, out_dtype, A.device)
    s = _stream_handle(stream)
    if plan is None:
        st = dgl_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), rows, ldc, K, m, n, out_dtype, s)
    else:
        st = dgl_gemm_planned(DTYPE_BF16, A.data_ptr(), B.data_ptr(), None, None, C.data_ptr(), rows, ldc, K,
                              m, n, out_dtype, plan, s)
    _check(st, "dgl_gemm_bf16")
    return C


def gemm_fp8(A, B, sa, sb, out=None, *, out_dtype=OUT_BF16, stream=None, plan: PlanInfo | None = None):
    """C = (A . B^T) * sa[:, None] * sb[None, :] for E4M3 A [m, K], B [n, K]; fp32 scales."""
    import torch
    _check_operand(A, "A", torch.float8_e4m3fn)
    _check_operand(B, "B", torch.float8_e4m3fn)
    m, K = A.shape
    n, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    for name, s_, length in (("sa", sa, m), ("sb", sb, n)):
        if s_.dtype != torch.float32 or not s_.is_cuda or s_.numel() != length or not s_.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of length {length}")
    C, ldc, rows = _out_tensor(out, m, n, out_dtype, A.device)
    s = _stream_handle(stream)
    if plan is None:
        st = dgl_gemm_fp8(A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), rows, ldc, K,
                          m, n, out_dtype, s)
    else:
        st = dgl_gemm_planned(DTYPE_E4M3, A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                              C.data_ptr(), rows, ldc, K, m, n, out_dtype, plan, s)
    _check(st, "dgl_gemm_fp8")
    return C


def gemm_mxfp4(A, B, sfa, sfb, K, out=None, *, out_dtype=OUT_BF16, stream=None):
    """C = sum_k 2^(sfa - 127) a * 2^(sfb - 127) b over E2M1 elements (MXFP4).

    A [m, K/2] and B [n, K/2] are uint8 CUDA tensors of packed E2M1 codes
    (element 2t in the low four bits of byte t); sfa [m, K/32] and sfb
    [n, K/32] are uint8 E8M0 scales, one per 32 elements of K.  K is passed
    explicitly (two elements per byte).  Returns C [m, n].
    """
    import torch
    m, n = A.shape[0], B.shape[0]
    for name, t, shape in (("A", A, (m, K // 2)), ("B", B, (n, K // 2)), ("sfa", sfa, (m, K // 32)),
                           ("sfb", sfb, (n, K // 32))):
        if t.dtype != torch.uint8 or not t.is_cuda or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor of shape {shape}")
    C, ldc, rows = _out_tensor(out, m, n, out_dtype, A.device)
    st = dgl_gemm_mxfp4(A.data_ptr(), B.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), C.data_ptr(), rows, ldc, K, m,
                        n, out_dtype, _stream_handle(stream))
    _check(st, "dgl_gemm_mxfp4")
    return C


def gemm_w4a8(A, B, sa, sb, K, out=None, *, out_dtype=OUT_BF16, stream=None):
    """C = (A . B^T) * sa[:, None] * sb[None, :] for E4M3 A [m, K] and E2M1 B.

    A is a float8_e4m3fn (or uint8) CUDA tensor [m, K]; B a uint8 CUDA tensor
    [n, K/2] of packed E2M1 codes (element 2t in the low four bits of byte t);
    sa [m], sb [n] fp32.  K is passed explicitly.  Returns C [m, n].
    """
    import torch
    m, n = A.shape[0], B.shape[0]
    if A.dtype not in (torch.float8_e4m3fn, torch.uint8) or not A.is_cuda or tuple(A.shape) != (m, K) \
            or not A.is_contiguous():
        raise ValueError(f"A must be a contiguous E4M3 CUDA tensor of shape {(m, K)}")
    if B.dtype != torch.uint8 or not B.is_cuda or tuple(B.shape) != (n, K // 2) or not B.is_contiguous():
        raise ValueError(f"B must be a contiguous uint8 CUDA tensor of shape {(n, K // 2)}")
    for name, s_, length in (("sa", sa, m), ("sb", sb, n)):
        if s_.dtype != torch.float32 or not s_.is_cuda or s_.numel() != length or not s_.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of length {length}")
    C, ldc, rows = _out_tensor(out, m, n, out_dtype, A.device)
    st = dgl_gemm_w4a8(A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), rows, ldc, K, m, n,
                       out_dtype, _stream_handle(stream))
    _check(st, "dgl_gemm_w4a8")
    return C


def plan(dtype, m, n, K, out_dtype=OUT_BF16, num_sms=0) -> dict:
    return dgl_plan(dtype, m, n, K, out_dtype, num_sms).as_dict()


def device_status(stream=None) -> int:
    return dgl_device_status(_stream_handle(stream))


def build() -> str:
    from ._build import build as _b
    return _b()


def linear(A, B, bias=None, out=None, *, act=ACT_NONE, gated=False, sa=None, sb=None, out_dtype=OUT_BF16,
           stream=None, plan: PlanInfo | None = None):
    """Linear layer with a fused epilogue: act(A . B^T + bias), or with
    gated=True act(A . Bg^T + bg) * (A . Bu^T + bu) for B = [Bg; Bu] (2n rows).

    A [m, K] and B are bf16 (or E4M3 with fp32 scales sa [m], sb [rows of B]);
    bias is fp32 with one entry per row of B, or None.  Returns C [m, n].
    """
    import torch
    e4m3 = A.dtype == torch.float8_e4m3fn
    want = torch.float8_e4m3fn if e4m3 else torch.bfloat16
    _check_operand(A, "A", want)
    _check_operand(B, "B", want)
    m, K = A.shape
    rows_b, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if gated and rows_b % 2:
        raise ValueError("a gated layer's B holds 2n rows: gate rows, then up rows")
    n = rows_b // 2 if gated else rows_b
    vecs = [("bias", bias, rows_b)] + ([("sa", sa, m), ("sb", sb, rows_b)] if e4m3 else [])
    for name, v, length in vecs:
        if v is None and name == "bias":
            continue
        if v is None or v.dtype != torch.float32 or not v.is_cuda or v.numel() != length or not v.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of length {length}")
    C, ldc, rows = _out_tensor(out, m, n, out_dtype, A.device)
    st = dgl_linear(DTYPE_E4M3 if e4m3 else DTYPE_BF16, A.data_ptr(), B.data_ptr(),
                    sa.data_ptr() if e4m3 else None, sb.data_ptr() if e4m3 else None,
                    bias.data_ptr() if bias is not None else None, C.data_ptr(), rows, ldc, K, m, n, out_dtype,
                    int(act), int(bool(gated)), plan, _stream_handle(stream))
    _check(st, "dgl_linear")
    return C

