"""W4A8 (E4M3 activations times packed E2M1 weights) through the C ABI, against
the oracle.

The GEMM guide's section 8.2 counts, for 4-bit weights, one byte per element
of A, half a byte per element of B and fp32 scales per row of A and of B.
dgl_gemm_w4a8 reads B's packed codes with TMA (16U4_ALIGN16B, which spreads
each 16 codes over a 16-byte unit of shared memory) and multiplies them on the
kind::f8f6f4 tensor cores beside E4M3 A.  Tolerance as every other product:
|C - C_ref| <= 1e-4 * S + 1e-6 (plus 1e-2 |C_ref| for bf16 output), and
integer-valued inputs exact.
"""
import numpy as np
import pytest
import torch

import dense_gemm_linear_gb300 as dgl
import oracle
from synthetic import make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _dev(case):
    A = torch.from_numpy(case.A).to(gu.DEV)
    B = torch.from_numpy(case.B).to(gu.DEV)
    return A, B, torch.from_numpy(case.sa).to(gu.DEV), torch.from_numpy(case.sb).to(gu.DEV)


def _run(case, *, guard_rows=0, pad_cols=0, plan=None, ops=None):
    A, B, sa, sb = ops if ops is not None else _dev(case)
    m, n, K = case.m, case.n, case.K
    rows, ldc = m + guard_rows, n + pad_cols
    Cbuf = gu.canary_buffer(rows, ldc, case.out)
    out_dtype = dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16
    s = torch.cuda.current_stream().cuda_stream
    if plan is None:
        st = dgl.dgl_gemm_w4a8(A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), Cbuf.data_ptr(), rows, ldc,
                               K, m, n, out_dtype, s)
    else:
        st = dgl.dgl_gemm_planned(dgl.DTYPE_W4A8, A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                                  Cbuf.data_ptr(), rows, ldc, K, m, n, out_dtype, plan, s)
    assert st == dgl.DGL_OK, dgl.status_string(st)
    st = dgl.dgl_device_status(s)
    assert st == dgl.DGL_OK, f"device status: {dgl.status_string(st)}"
    bits = Cbuf.view(torch.int32) if case.out == "f32" else Cbuf.view(torch.int16)
    canary = gu.CANARY_F32 if case.out == "f32" else gu.CANARY_BF16
    intact = bool((bits[m:, :] == canary).all().item()) and bool((bits[:m, n:] == canary).all().item())
    return Cbuf, intact


def _check_full(case, Cbuf):
    ref, S = oracle.w4a8_gemm(case.A, case.B, case.sa, case.sb)
    got = Cbuf[:case.m, :case.n].double().cpu().numpy()
    gu._assert_within(case, got, ref, S, "full compare")


def _check_exact(case, Cbuf):
    ref, _ = oracle.w4a8_gemm(case.A, case.B, case.sa, case.sb)
    got = Cbuf[:case.m, :case.n].double().cpu().numpy()
    assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref), "reference not exact in fp32"
    mism = got != ref
    assert not mism.any(), f"{int(mism.sum())} elements differ; first {np.argwhere(mism)[:4].tolist()}"


def _check_sampled(case, Cbuf, tile_m=256, tile_n=256):
    rows, cols = gu.sample_points(case, tile_m, tile_n, seed=case.seed)
    ref, S = oracle.w4a8_gemm_points(case.A, case.B, case.sa, case.sb, rows, cols)
    got = Cbuf[torch.from_numpy(rows).to(Cbuf.device), torch.from_numpy(cols).to(Cbuf.device)].double().cpu().numpy()
    gu._assert_within(case, got, ref, S, "sampled points")


@pytest.mark.parametrize("m", [1, 5, 16, 17, 200, 300])
def test_w4a8_integer_exact(m):
    """Integer E4M3 times any E2M1 code, scales in {1/2, 1, 2}: exact in fp32,
    on the decode path (m <= 16) and the tile path."""
    case = make_case("w4a8", m, 300, 512, out="f32", dist="int")
    Cbuf, intact = _run(case, guard_rows=2, pad_cols=3)
    assert intact
    _check_exact(case, Cbuf)


@pytest.mark.parametrize("m,n,k", [(130, 200, 128), (1, 37, 256), (16, 1000, 1024), (333, 517, 384),
                                   (600, 700, 2048), (8, 4096, 4096)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_w4a8_general(m, n, k, out):
    case = make_case("w4a8", m, n, k, out=out, dist="w4a8")
    Cbuf, intact = _run(case, guard_rows=3, pad_cols=5)
    assert intact, "wrote outside the valid region"
    _check_full(case, Cbuf)


LADDER = [(64, 64), (64, 256), (128, 64), (128, 128), (128, 256), (256, 128), (256, 256)]


@pytest.mark.parametrize("tm,tn", LADDER)
def test_w4a8_every_rung(tm, tn):
    """Each tile of the ladder on a shape none of them divides."""
    case = make_case("w4a8", 333, 517, 384, out="bf16", dist="w4a8")
    Cbuf, intact = _run(case, guard_rows=4, pad_cols=7, plan=dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm, tile_n=tn))
    assert intact
    _check_full(case, Cbuf)


def test_w4a8_stream_k_and_split_tail_exact():
    """The tile kernel's other schedules with 4-bit B: stream-K partial tiles and
    the half tiles of a split tail (half-height 4-bit B boxes)."""
    case = make_case("w4a8", 900, 1100, 2048, out="f32", dist="int")
    ops = _dev(case)
    for plan in (dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, stream_k=1),
                 dgl.PlanInfo(path=dgl.PATH_TC, tile_m=128, tile_n=256, stream_k=1)):
        Cbuf, intact = _run(case, plan=plan, ops=ops)
        assert intact
        _check_exact(case, Cbuf)
    case = make_case("w4a8", 4000, 4200, 1024, out="f32", dist="int")
    Cbuf, intact = _run(case, plan=dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, split_tail=1))
    assert intact
    _check_sampled(case, Cbuf)


@pytest.mark.parametrize("m,n,k", [(597, 11008, 4096), (16, 11008, 4096), (1, 11008, 4096)])
def test_w4a8_llama_shapes_sampled(m, n, k):
    """The LLaMA-2 7B up/gate shapes at full size: a seeded sample and whole
    corner tiles against the oracle."""
    case = make_case("w4a8", m, n, k, out="bf16", dist="w4a8")
    Cbuf, intact = _run(case, guard_rows=1)
    assert intact
    _check_sampled(case, Cbuf)


def test_w4a8_argument_errors():
    case = make_case("w4a8", 64, 64, 256, out="f32", dist="int")
    A, B, sa, sb = _dev(case)
    C = torch.empty((64, 64), dtype=torch.float32, device=gu.DEV)
    s = torch.cuda.current_stream().cuda_stream

    def call(a, b, K):
        return dgl.dgl_gemm_w4a8(a, b, sa.data_ptr(), sb.data_ptr(), C.data_ptr(), 64, 64, K, 64, 64,
                                 dgl.OUT_F32, s)
    assert call(A.data_ptr(), B.data_ptr(), 192) == dgl.DGL_ERR_ALIGN          # K not a multiple of 128
    Bpad = torch.zeros(B.numel() + 16, dtype=torch.uint8, device=gu.DEV)
    assert call(A.data_ptr(), Bpad.data_ptr() + 16, 256) == dgl.DGL_ERR_ALIGN  # B 16- but not 32-byte aligned
    assert dgl.dgl_gemm_w4a8(A.data_ptr(), B.data_ptr(), None, sb.data_ptr(), C.data_ptr(), 64, 64, 256, 64, 64,
                             dgl.OUT_F32, s) == dgl.DGL_ERR_ARG
    assert call(A.data_ptr(), B.data_ptr(), 256) == dgl.DGL_OK
    torch.cuda.synchronize()


def test_w4a8_torch_helper():
    case = make_case("w4a8", 40, 300, 256, out="f32", dist="w4a8")
    A, B, sa, sb = _dev(case)
    C = dgl.gemm_w4a8(A.view(torch.float8_e4m3fn), B, sa, sb, case.K, out_dtype=dgl.OUT_F32)
    assert dgl.device_status() == dgl.DGL_OK
    ref, S = oracle.w4a8_gemm(case.A, case.B, case.sa, case.sb)
    gu._assert_within(case, C.double().cpu().numpy(), ref, S, "torch helper")
