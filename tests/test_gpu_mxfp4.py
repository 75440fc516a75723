"""Block-scaled FP4 (MXFP4, dgl_gemm_mxfp4) vs the oracle, through the C ABI.

C[i, j] = sum_k 2^(sfa[i][k/32] - 127) a(i, k) * 2^(sfb[j][k/32] - 127) b(j, k)
with E2M1 elements packed two to a byte.  Tolerance as in the other parity
tests: |C - C_ref| <= 1e-4 * sum_k |a b| (scaled) + 1e-6 for fp32 output,
plus 1e-2 |C_ref| for bf16 output.  The integer recipe (magnitudes <= 3,
scales 2^-1 .. 2^1) makes every partial sum a multiple of 2^-4 below 2^24
quanta, so fp32 output must equal the oracle exactly and bf16 output its
round-to-nearest-even.  Every case also checks that nothing outside the
valid region of C was written (guard rows and padded pitch of canaries).
"""
import numpy as np
import pytest
import torch

import dense_gemm_linear_gb300 as dgl
import oracle
from synthetic import make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _dev(case, scale_offset=0):
    A = torch.from_numpy(case.A).cuda()
    B = torch.from_numpy(case.B).cuda()
    # scales copied at a byte offset into a larger buffer when asked, so the
    # kernel's 8-byte scale reads cannot be used
    def sc(x):
        if not scale_offset:
            return torch.from_numpy(x).cuda(), None
        buf = torch.zeros(x.size + 64, dtype=torch.uint8, device="cuda")
        buf[scale_offset:scale_offset + x.size] = torch.from_numpy(x.ravel()).cuda()
        return buf, buf[scale_offset:].data_ptr()
    sa, pa = sc(case.sa)
    sb, pb = sc(case.sb)
    return A, B, (sa, pa), (sb, pb)


def _run(case, *, guard_rows=0, pad_cols=0, scale_offset=0):
    A, B, (sa, pa), (sb, pb) = _dev(case, scale_offset)
    m, n, K = case.m, case.n, case.K
    rows, ldc = m + guard_rows, n + pad_cols
    Cbuf = gu.canary_buffer(rows, ldc, case.out)
    out_dtype = dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16
    s = torch.cuda.current_stream().cuda_stream
    st = dgl.dgl_gemm_mxfp4(A.data_ptr(), B.data_ptr(), pa or sa.data_ptr(), pb or sb.data_ptr(), Cbuf.data_ptr(),
                            rows, ldc, K, m, n, out_dtype, s)
    assert st == dgl.DGL_OK, dgl.status_string(st)
    st = dgl.dgl_device_status(s)
    assert st == dgl.DGL_OK, f"device status: {dgl.status_string(st)}"
    bits = Cbuf.view(torch.int32) if case.out == "f32" else Cbuf.view(torch.int16)
    canary = gu.CANARY_F32 if case.out == "f32" else gu.CANARY_BF16
    intact = bool((bits[m:, :] == canary).all().item()) and bool((bits[:m, n:] == canary).all().item())
    assert intact, f"{case.name}: wrote outside the valid region"
    return Cbuf


def _close(case, got, ref, S, where="full"):
    assert np.isfinite(got).all(), f"{case.name}: non-finite output"
    bound = (1e-2 if case.out == "bf16" else 0.0) * np.abs(ref) + 1e-4 * S + 1e-6
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{case.name}: {int(bad.sum())} of {bad.size} out of tolerance at {where} "
                             f"(max err {float(err.max()):.3e}); first "
                             f"{[(tuple(map(int, i)), float(got[tuple(i)]), float(ref[tuple(i)])) for i in idx]}")


def _exact(case, got, ref):
    if case.out == "f32":
        assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref), "reference not exact in fp32"
        mism = got != ref
    else:
        want = oracle.round_bf16(ref)
        have = torch.from_numpy(got.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        mism = have != want
    if mism.any():
        idx = np.argwhere(mism)[:5]
        raise AssertionError(f"{case.name}: {int(mism.sum())} elements differ from the exact result; first "
                             f"{[(tuple(map(int, i)), float(got[tuple(i)]), float(ref[tuple(i)])) for i in idx]}")


def _full(case, **kw):
    Cbuf = _run(case, **kw)
    got = Cbuf[:case.m, :case.n].double().cpu().numpy()
    ref, S = oracle.mxfp4_gemm(case.A, case.B, case.sa, case.sb)
    if case.dist == "int":
        _exact(case, got, ref)
    else:
        _close(case, got, ref, S)


# ------------------------------------------------------------ one tile first
def test_one_tile_one_instruction():
    """128 x 256 x 64: a single tile, one K = 64 step (two scale blocks) per 128-column half."""
    _full(make_case("mxfp4", 128, 256, 64, out="f32", dist="int"))


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("m,n,k", [(128, 128, 256), (200, 300, 512), (333, 517, 1024), (129, 257, 2048)])
def test_integer_exact(m, n, k, out):
    """Whole stages (K a multiple of 256: 8-byte scale reads), ragged m and n."""
    _full(make_case("mxfp4", m, n, k, out=out, dist="int"), guard_rows=2, pad_cols=3)


@pytest.mark.parametrize("k", [32, 96, 224, 800, 4064])
def test_ragged_k(k):
    """K not a multiple of a stage: a partial last stage, byte-wise scale reads,
    blocks past K read as scale 1 beside zero-filled elements."""
    _full(make_case("mxfp4", 190, 260, k, out="f32", dist="int"), guard_rows=1, pad_cols=1)


@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("m,n,k", [(256, 256, 512), (300, 517, 1024), (1000, 700, 4096)])
def test_quantised_normal(m, n, k, out):
    """OCP MX block quantisation of N(0,1) activations and N(0, 0.02^2) weights."""
    _full(make_case("mxfp4", m, n, k, out=out, dist="mx"), guard_rows=1, pad_cols=5)


def test_unaligned_scale_pointers():
    """Scale arrays at odd byte offsets: the kernel reads them byte by byte."""
    _full(make_case("mxfp4", 260, 140, 512, out="f32", dist="int"), scale_offset=3)


@pytest.mark.parametrize("m", [1, 5, 16, 17])
def test_small_m(m):
    """Few rows of A (no decode path for MXFP4): one partial row tile."""
    _full(make_case("mxfp4", m, 1000, 1024, out="f32", dist="int"), guard_rows=1)


def test_persistent_many_tiles_and_repeat():
    """More tiles than SMs (a CTA walks several, reusing its accumulator and
    the whole scale ring), and two calls in a row give the same bits."""
    case = make_case("mxfp4", 2560, 2048, 256, out="f32", dist="int")  # 20 x 8 = 160 tiles of 128 x 256
    C1 = _run(case)
    C2 = _run(case)
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))
    ref, _ = oracle.mxfp4_gemm(case.A, case.B, case.sa, case.sb)
    _exact(case, C1[:case.m, :case.n].double().cpu().numpy(), ref)


def test_full_size_sampled():
    """4096 x 4096 x 4096 with quantised normal inputs, checked on a seeded
    sample plus full tiles at the edges."""
    case = make_case("mxfp4", 4096, 4096, 4096, out="bf16", dist="mx")
    Cbuf = _run(case)
    rows, cols = gu.sample_points(case, 128, 256, seed=5)
    ref, S = oracle.mxfp4_gemm_points(case.A, case.B, case.sa, case.sb, rows, cols)
    got = Cbuf[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    _close(case, got, ref, S, "sampled points")


def test_k_zero_and_empty():
    case = make_case("mxfp4", 40, 50, 32, out="f32", dist="int")
    A, B, (sa, _), (sb, _) = _dev(case)
    C = gu.canary_buffer(40, 50, "f32")
    s = torch.cuda.current_stream().cuda_stream
    assert dgl.dgl_gemm_mxfp4(A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), 40, 50, 0,
                              40, 50, dgl.OUT_F32, s) == dgl.DGL_OK
    assert dgl.dgl_device_status(s) == dgl.DGL_OK
    assert bool((C == 0).all().item())
    assert dgl.dgl_gemm_mxfp4(A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), 40, 50, 32,
                              40, 0, dgl.OUT_F32, s) == dgl.DGL_OK  # n_valid 0 -> N: a full product


def test_argument_errors():
    case = make_case("mxfp4", 64, 64, 64, out="bf16", dist="int")
    A, B, (sa, _), (sb, _) = _dev(case)
    C = torch.empty(64, 64, device="cuda", dtype=torch.bfloat16)
    s = torch.cuda.current_stream().cuda_stream

    def call(a=A.data_ptr(), sfa=sa.data_ptr(), k=64, out=dgl.OUT_BF16):
        return dgl.dgl_gemm_mxfp4(a, B.data_ptr(), sfa, sb.data_ptr(), C.data_ptr(), 64, 64, k, 64, 64, out, s)

    assert call(k=48) == dgl.DGL_ERR_ALIGN           # not whole 32-element blocks
    assert call(sfa=None) == dgl.DGL_ERR_ARG
    assert call(a=A.data_ptr() + 8) == dgl.DGL_ERR_ALIGN
    assert call(out=7) == dgl.DGL_ERR_ARG
    assert call() == dgl.DGL_OK
    assert dgl.dgl_device_status(s) == dgl.DGL_OK
