"""The backward-pass operand layouts (dgl_gemm_bf16_ex) vs the oracle, through the C ABI.

A linear layer's training step runs three GEMMs on the same row-major
tensors ("GEMM analysis in TraceLens", sections "Backward pass GEMMs" and
"How PyTorch calls BLAS"): Y = X W^T (both operands K-major), dX = dY W
(B = W stored [K][n], MN-major) and dW = dY^T X (both MN-major).  The oracle
computes the same product from K-major copies of the operands.  Tolerance as
in the other parity tests: |C - C_ref| <= 1e-4 sum_k |a b| + 1e-6 (fp32 C),
plus 1e-2 |C_ref| for bf16 C; integer-valued inputs must match exactly.
"""
import numpy as np
import pytest
import torch

import dense_gemm_linear_gb300 as dgl
from synthetic import make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

K_, MN_ = dgl.K_MAJOR, dgl.MN_MAJOR


def _stored(codes, major, extra):
    """Device bf16 tensor holding `codes` ([rows][K]) K-major, or its transpose
    MN-major, in a buffer whose row pitch is the packed one rounded up to a
    multiple of 8 elements, plus `extra` (a multiple of 8)."""
    x = codes if major == K_ else np.ascontiguousarray(codes.T)
    rows, cols = x.shape
    pitch = -(-cols // 8) * 8 + extra
    buf = np.zeros((rows, pitch), dtype=np.uint16)
    buf[:, :cols] = x
    t = torch.from_numpy(buf.view(np.int16)).view(torch.bfloat16).cuda()
    return t, pitch


def _run(case, a_major, b_major, *, pad_a=0, pad_b=0, pad_c=0, plan=None):
    A, lda = _stored(case.A, a_major, pad_a)
    B, ldb = _stored(case.B, b_major, pad_b)
    m, n, K = case.m, case.n, case.K
    ldc = n + pad_c
    Cbuf = gu.canary_buffer(m + 1, ldc, case.out)
    out = dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16
    s = torch.cuda.current_stream().cuda_stream
    st = dgl.dgl_gemm_bf16_ex(a_major, b_major, A.data_ptr(), lda, B.data_ptr(), ldb, Cbuf.data_ptr(), ldc, m, n, K,
                              out, plan, s)
    assert st == dgl.DGL_OK, dgl.status_string(st)
    st = dgl.dgl_device_status(s)
    assert st == dgl.DGL_OK, f"device status: {dgl.status_string(st)}"
    bits = Cbuf.view(torch.int32) if case.out == "f32" else Cbuf.view(torch.int16)
    canary = gu.CANARY_F32 if case.out == "f32" else gu.CANARY_BF16
    assert bool((bits[m:, :] == canary).all().item()) and bool((bits[:m, n:] == canary).all().item()), \
        "wrote outside the valid region"
    return Cbuf


LAYOUTS = [(K_, MN_), (MN_, MN_), (MN_, K_), (K_, K_)]
TILES = [(128, 64), (128, 128), (128, 256), (256, 128), (256, 256)]


@pytest.mark.parametrize("layout", LAYOUTS, ids=["dX", "dW", "A_mn", "pitched"])
@pytest.mark.parametrize("tile", TILES, ids=lambda t: f"{t[0]}x{t[1]}")
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_layouts_every_tile(layout, tile, out):
    """m, n and K all ragged against the tiles and the 64-wide boxes; padded pitches."""
    case = make_case("bf16", 300, 260, 200, out=out)
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tile[0], tile_n=tile[1])
    Cbuf = _run(case, *layout, pad_a=8, pad_b=16, pad_c=3, plan=plan)
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("layout", LAYOUTS, ids=["dX", "dW", "A_mn", "pitched"])
def test_layouts_integer_exact(layout):
    case = make_case("bf16", 257, 320, 384, out="f32", dist="int")
    Cbuf = _run(case, *layout, pad_a=8, pad_b=8)
    gu.assert_exact(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("m", [1, 16])
def test_layouts_small_m_take_the_tile_path(m):
    case = make_case("bf16", m, 520, 256, out="f32")
    Cbuf = _run(case, MN_, MN_, pad_a=8)
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("layout", [(K_, MN_), (MN_, MN_)], ids=["dX", "dW"])
def test_layouts_split_tail(layout):
    case = make_case("bf16", 2304, 2304, 256, out="bf16")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, split_tail=1)
    Cbuf = _run(case, *layout, plan=plan)
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


def test_layouts_stream_k():
    case = make_case("bf16", 600, 1100, 1024, out="f32")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, stream_k=1)
    Cbuf = _run(case, MN_, MN_, plan=plan)
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("which", ["dX", "dW"])
def test_gpt3xl_backward_full_size(which):
    """GPT-3-XL (d_model 2048, d_ff 8192, 5 x 2048 tokens): the backward GEMMs
    10240 x 2048 x 8192 (dX) and 8192 x 2048 x 10240 (dW), sampled."""
    if which == "dX":
        case = make_case("bf16", 10240, 2048, 8192, out="bf16")
        layout = (K_, MN_)
    else:
        case = make_case("bf16", 8192, 2048, 10240, out="bf16")
        layout = (MN_, MN_)
    Cbuf = _run(case, *layout)
    gu.assert_close_sampled(case, Cbuf, tile_m=256, tile_n=256, seed=11)


def test_layout_argument_errors():
    case = make_case("bf16", 64, 64, 64, out="bf16")
    A, lda = _stored(case.A, MN_, 0)
    B, ldb = _stored(case.B, MN_, 0)
    C = torch.empty(64, 64, device="cuda", dtype=torch.bfloat16)
    s = torch.cuda.current_stream().cuda_stream

    def call(a_major=MN_, b_major=MN_, lda_=lda, ldb_=ldb):
        return dgl.dgl_gemm_bf16_ex(a_major, b_major, A.data_ptr(), lda_, B.data_ptr(), ldb_, C.data_ptr(), 64, 64,
                                    64, 64, dgl.OUT_BF16, None, s)

    assert call(a_major=2) == dgl.DGL_ERR_ARG
    assert call(lda_=56) == dgl.DGL_ERR_ARG        # shorter than the row's extent
    assert call(lda_=68) == dgl.DGL_ERR_ALIGN      # 136 bytes: not a multiple of 16
    assert call() == dgl.DGL_OK
    assert dgl.dgl_device_status(s) == dgl.DGL_OK
