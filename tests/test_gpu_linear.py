"""Linear-layer epilogue (dgl_linear) vs the oracle, element by element, through the C ABI.

C = act(A . B^T + bias), and the gated form act(A . Bg^T + bg) * (A . Bu^T + bu)
with B = [Bg; Bu].  Tolerance: |C - C_ref| <= 1e-2 |C_ref| (bf16 output)
+ 1e-4 E + 1e-6, where E is the oracle's error scale: the product's own
allowance (1e-4 of sum_k |a b| plus |bias|) carried through the activation
(slope at most 1.2) and, when gated, through the product of the two halves.
Every case also checks that nothing outside the valid region of C was written.
"""
import numpy as np
import pytest
import torch

import dense_gemm_linear_gb300 as dgl
import oracle
from synthetic import make_case, normal
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

STREAM_BIAS = 4
ACTS = {"none": dgl.ACT_NONE, "gelu": dgl.ACT_GELU, "silu": dgl.ACT_SILU}


def _bias(rows, seed=0):
    return normal(seed, STREAM_BIAS, (rows,), 0.0, 0.5).astype(np.float32)


def _case(dtype, m, n, k, out, gated, dist=None):
    rows_b = 2 * n if gated else n
    case = make_case(dtype, m, rows_b, k, out=out, dist=dist or ("fp8" if dtype == "fp8" else "normal"))
    case.n = n  # the output's columns; B keeps its 2n rows when gated
    return case


def _run(case, bias, act, gated, *, plan=None, guard_rows=0, pad_cols=0):
    A, B, sa, sb = gu.to_device(case)
    m, n, K = case.m, case.n, case.K
    rows, ldc = m + guard_rows, n + pad_cols
    Cbuf = gu.canary_buffer(rows, ldc, case.out)
    bias_t = torch.from_numpy(bias).cuda() if bias is not None else None
    out_dtype = dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16
    s = torch.cuda.current_stream().cuda_stream
    st = dgl.dgl_linear(dgl.DTYPE_BF16 if case.dtype == "bf16" else dgl.DTYPE_E4M3, A.data_ptr(), B.data_ptr(),
                        sa.data_ptr() if sa is not None else None, sb.data_ptr() if sb is not None else None,
                        bias_t.data_ptr() if bias_t is not None else None, Cbuf.data_ptr(), rows, ldc, K, m, n,
                        out_dtype, act, int(gated), plan, s)
    assert st == dgl.DGL_OK, dgl.status_string(st)
    st = dgl.dgl_device_status(s)
    assert st == dgl.DGL_OK, f"device status: {dgl.status_string(st)}"
    bits = Cbuf.view(torch.int32) if case.out == "f32" else Cbuf.view(torch.int16)
    canary = gu.CANARY_F32 if case.out == "f32" else gu.CANARY_BF16
    intact = bool((bits[m:, :] == canary).all().item()) and bool((bits[:m, n:] == canary).all().item())
    assert intact, "wrote outside the valid region"
    return Cbuf


def _ref(case, bias, act, gated, rows=None, cols=None):
    dt = oracle.BF16 if case.dtype == "bf16" else oracle.E4M3
    if rows is None:
        return oracle.linear(dt, case.A, case.B, case.sa, case.sb, bias=bias, act=act, gated=gated)
    return oracle.linear_points(dt, case.A, case.B, rows, cols, case.sa, case.sb, bias=bias, act=act, gated=gated)


def _within(case, got, ref, E, where=""):
    assert np.isfinite(got).all(), "non-finite output"
    bound = (1e-2 if case.out == "bf16" else 0.0) * np.abs(ref) + 1e-4 * E + 1e-6
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} out of tolerance {where} (max err {err.max():.3e}); "
                             f"first {[(tuple(map(int, i)), float(got[tuple(i)]), float(ref[tuple(i)])) for i in idx]}")


def _full(case, bias, act, gated, **kw):
    Cbuf = _run(case, bias, act, gated, **kw)
    got = Cbuf[:case.m, :case.n].double().cpu().numpy()
    ref, E = _ref(case, bias, act, gated)
    _within(case, got, ref, E)


# ------------------------------------------------------------ bias and activation
@pytest.mark.parametrize("act", sorted(ACTS))
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("with_bias", [True, False])
def test_bias_activation(act, out, with_bias):
    case = _case("bf16", 300, 517, 136, out, False)
    bias = _bias(517) if with_bias else None
    _full(case, bias, ACTS[act], False, guard_rows=2, pad_cols=3)


@pytest.mark.parametrize("tile", [(128, 128), (128, 256), (256, 128), (256, 256)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_every_linear_tile(tile, out):
    """Every tile with a linear-layer variant; n = 517 ends inside a 16-byte unit."""
    case = _case("bf16", 300, 517, 200, out, False)
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tile[0], tile_n=tile[1])
    _full(case, _bias(517), dgl.ACT_GELU, False, plan=plan, guard_rows=1, pad_cols=2)


@pytest.mark.parametrize("m", [1, 5, 16])
def test_decode_bias_activation(m):
    case = _case("bf16", m, 777, 520, "bf16", False)
    assert dgl.dgl_plan(0, m, 777, 520).path == dgl.PATH_DECODE
    _full(case, _bias(777), dgl.ACT_SILU, False, guard_rows=1, pad_cols=1)


@pytest.mark.parametrize("dtype,k", [("bf16", 512), ("fp8", 1024)])
def test_decode_stacked_bias_activation(dtype, k):
    """The decode epilogue after the G-slot sum (777 columns in parts of 6 rows: G = 8)."""
    case = _case(dtype, 5, 777, k, "bf16", False)
    assert dgl.dgl_plan(0 if dtype == "bf16" else 1, 5, 777, k).k_group == 8
    _full(case, _bias(777), dgl.ACT_GELU, False, guard_rows=1, pad_cols=1)


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_e4m3_scaled_bias_activation(act):
    case = _case("fp8", 260, 384, 256, "bf16", False)
    _full(case, _bias(384), ACTS[act], False, pad_cols=8)


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_activation_accuracy_over_a_wide_range(act):
    """A = I makes C = act(B^T + bias) exactly up to the activation, so the
    kernel's activation is checked against the oracle's fp64 one directly:
    inputs beyond +-10, error within 4e-6 |x| + 1e-6."""
    K = 128
    case = _case("bf16", K, 640, K, "f32", False)
    from synthetic import to_bf16_codes
    case.A = to_bf16_codes(np.eye(K))
    case.B = to_bf16_codes(normal(1, 1, (640, K), 0.0, 3.0))
    bias = np.linspace(-6.0, 6.0, 640).astype(np.float32)
    Cbuf = _run(case, bias, ACTS[act], False)
    got = Cbuf[:K, :640].double().cpu().numpy()
    ref, _ = _ref(case, bias, ACTS[act], False)
    x = gu.oracle.decode_bf16(case.B).T + bias[None, :].astype(np.float64)
    assert np.abs(x).max() > 10.0
    err = np.abs(got - ref)
    assert (err <= 4e-6 * np.abs(x) + 1e-6).all(), f"max err {err.max():.3e}"


def test_split_tail_with_linear_epilogue():
    """The last wave's half tiles take the bias and activation too."""
    case = _case("bf16", 2304, 2304, 256, "bf16", False)
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, split_tail=1)
    _full(case, _bias(2304), dgl.ACT_GELU, False, plan=plan, pad_cols=2)


# ------------------------------------------------------------ gated up projection
@pytest.mark.parametrize("act", ["gelu", "silu", "none"])
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("tile_n", [128, 256])
def test_gated(act, out, tile_n):
    n = 333  # ragged in both tile widths; bf16 rows of 666 bytes are not 16-byte aligned
    case = _case("bf16", 300, n, 200, out, True)
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=tile_n)
    _full(case, _bias(2 * n), ACTS[act], True, plan=plan, guard_rows=2, pad_cols=1)


@pytest.mark.parametrize("m", [1, 3, 17])
def test_gated_small_m_runs_on_pairs(m):
    case = _case("bf16", m, 512, 256, "bf16", True)
    _full(case, None, dgl.ACT_SILU, True, guard_rows=1)


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_gated_e4m3_scales(act):
    """The up half takes the scales and bias of rows n .. 2n-1 of B."""
    case = _case("fp8", 200, 384, 512, "bf16", True)
    _full(case, _bias(768), ACTS[act], True)


def test_gated_integer_exact():
    """Integer inputs, identity activation: gate * up is exact in fp32."""
    case = _case("bf16", 260, 300, 64, "f32", True, dist="int")
    Cbuf = _run(case, None, dgl.ACT_NONE, True)
    got = Cbuf[:case.m, :case.n].double().cpu().numpy()
    ref, _ = _ref(case, None, dgl.ACT_NONE, True)
    assert np.array_equal(got, ref)


def test_gated_llama_up_gate_full_size():
    """The LLaMA-2 7B prefill up/gate pair as one call: 597 x 11008 x 4096, B of 22016 rows."""
    case = _case("bf16", 597, 11008, 4096, "bf16", True)
    Cbuf = _run(case, None, dgl.ACT_SILU, True)
    rows, cols = gu.sample_points(case, 256, 128, seed=3)
    ref, E = _ref(case, None, dgl.ACT_SILU, True, rows, cols)
    got = Cbuf[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    _within(case, got, ref, E, "at sampled points")


# ------------------------------------------------------------ errors
def test_linear_argument_errors():
    case = _case("bf16", 64, 128, 64, "bf16", True)
    A, B, _, _ = gu.to_device(case)
    C = torch.empty(64, 128, device="cuda", dtype=torch.bfloat16)
    s = torch.cuda.current_stream().cuda_stream

    def call(act=dgl.ACT_SILU, gated=1, plan=None):
        return dgl.dgl_linear(dgl.DTYPE_BF16, A.data_ptr(), B.data_ptr(), None, None, None, C.data_ptr(), 64, 128,
                              64, 64, 128, dgl.OUT_BF16, act, gated, plan, s)

    assert call(act=3) == dgl.DGL_ERR_ARG
    assert call(gated=2) == dgl.DGL_ERR_ARG
    # a gated layer needs a CTA-pair tile; 64-wide tiles have no linear variant
    assert call(plan=dgl.PlanInfo(path=dgl.PATH_TC, tile_m=128, tile_n=256)) == dgl.DGL_ERR_UNSUPPORTED
    assert call(gated=0, plan=dgl.PlanInfo(path=dgl.PATH_TC, tile_m=128, tile_n=64)) == dgl.DGL_ERR_UNSUPPORTED
    assert call(plan=dgl.PlanInfo(path=dgl.PATH_DECODE)) == dgl.DGL_ERR_UNSUPPORTED
    assert dgl.dgl_device_status(s) == dgl.DGL_OK
