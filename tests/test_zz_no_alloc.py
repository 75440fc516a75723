"""dgl_gemm_noalloc: the GEMM entry point that allocates no device memory.

Some callers cannot call cudaMalloc while they run: a framework that owns all
device memory through its own pool, or a serving loop that allows no
allocation after start-up.  dgl_gemm_noalloc serves them by keeping its
stream-K partial tiles in a fixed device array instead of a workspace it
allocates.  These tests call it through the C ABI on problems whose last wave
is split (so the array is really used) and compare each of two calls in a row
with the existing entry point (dgl_gemm_bf16 / dgl_gemm_fp8) and with the
oracle (a seeded sample plus whole corner tiles): within the parity tolerance
|C - C_ref| <= 1e-4 * sum_k |a_ik b_jk| + 1e-6 (plus 1e-2 |C_ref| for bf16
output), and bit for bit on integer-valued inputs.  One test checks that a
call leaves the device's free memory unchanged while the allocating stream-K
path does not.  The file is named to run last.
"""
import math

import numpy as np
import pytest
import torch

import dense_gemm_linear_gb300 as dgl
from synthetic import make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _split_last_wave(case, out_dtype):
    """True when the planner's tile leaves a partial last wave that stream-K splits."""
    dtype = dgl.DTYPE_BF16 if case.dtype == "bf16" else dgl.DTYPE_E4M3
    num_sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = dgl.dgl_plan(dtype, case.m, case.n, case.K, out_dtype, num_sms)
    if plan.path != dgl.PATH_TC:
        return False
    tiles = math.ceil(case.m / plan.tile_m) * math.ceil(case.n / plan.tile_n)
    units = num_sms // plan.cta_group
    nk = math.ceil(case.K * (1 if case.dtype == "fp8" else 2) / 128)
    tail = tiles % units
    return tail != 0 and tail * nk >= 4 * units


def _call(case, A, B, sa, sb, noalloc):
    """One call into a canary-filled C; returns (C, canaries intact)."""
    m, n, K = case.m, case.n, case.K
    out_dtype = dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16
    C = gu.canary_buffer(m + 3, n, case.out)  # three guard rows
    s = torch.cuda.current_stream().cuda_stream
    sa_p = sa.data_ptr() if sa is not None else None
    sb_p = sb.data_ptr() if sb is not None else None
    if noalloc:
        dtype = dgl.DTYPE_BF16 if case.dtype == "bf16" else dgl.DTYPE_E4M3
        st = dgl.dgl_gemm_noalloc(dtype, A.data_ptr(), B.data_ptr(), sa_p, sb_p, C.data_ptr(),
                                  m + 3, n, K, m, n, out_dtype, s)
    elif case.dtype == "bf16":
        st = dgl.dgl_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), m + 3, n, K, m, n, out_dtype, s)
    else:
        st = dgl.dgl_gemm_fp8(A.data_ptr(), B.data_ptr(), sa_p, sb_p, C.data_ptr(), m + 3, n, K, m, n,
                              out_dtype, s)
    assert st == dgl.DGL_OK, dgl.status_string(st)
    st = dgl.dgl_device_status(s)
    assert st == dgl.DGL_OK, f"device status: {dgl.status_string(st)}"
    bits = C.view(torch.int32) if case.out == "f32" else C.view(torch.int16)
    canary = gu.CANARY_F32 if case.out == "f32" else gu.CANARY_BF16
    intact = bool((bits[m:, :] == canary).all().item())
    return C[:m], intact


def _abs_sum(case, A, B, sa, sb):
    """S[i, j] = sum_k |a_ik b_jk| (times |sa_i sb_j|), in fp64 on the device."""
    S = A.double().abs() @ B.double().abs().T
    if sa is not None:
        S = S * (sa.double().abs()[:, None] * sb.double().abs()[None, :])
    return S


CASES = [
    ("bf16", 2048, 11007, 1024, "bf16", "normal"),  # ragged n: the row-staging epilogue
    ("fp8", 597, 11008, 4096, "bf16", "fp8"),      # the LLaMA up/gate shape in E4M3
    ("bf16", 1800, 7000, 2048, "f32", "normal"),
]


@pytest.mark.parametrize("dtype,m,n,k,out,dist", CASES)
def test_noalloc_matches_existing_entry_point(dtype, m, n, k, out, dist):
    case = make_case(dtype, m, n, k, out=out, dist=dist)
    out_dtype = dgl.OUT_F32 if out == "f32" else dgl.OUT_BF16
    assert _split_last_wave(case, out_dtype), "test setup: this shape should split its last wave"
    A, B, sa, sb = gu.to_device(case)
    ref, intact = _call(case, A, B, sa, sb, noalloc=False)
    assert intact
    ref = ref.double()
    bound = (1e-2 if out == "bf16" else 0.0) * ref.abs() + 1e-4 * _abs_sum(case, A, B, sa, sb) + 1e-6
    plan = dgl.dgl_plan(dgl.DTYPE_BF16 if dtype == "bf16" else dgl.DTYPE_E4M3, m, n, k, out_dtype)
    for call in range(2):  # the second call finds the array as the first one left it
        got, intact = _call(case, A, B, sa, sb, noalloc=True)
        assert intact, f"call {call}: wrote outside the valid region"
        # against the oracle: a seeded sample and whole tiles at every corner
        gu.assert_close_sampled(case, got, plan.tile_m, plan.tile_n, seed=call)
        got = got.double()
        assert torch.isfinite(got).all(), f"call {call}: non-finite output"
        err = (got - ref).abs()
        bad = int((err > bound).sum().item())
        assert bad == 0, f"call {call}: {bad} elements out of tolerance (max err {float(err.max()):.3e})"


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_noalloc_integer_inputs_bit_exact(dtype):
    """Integer-valued inputs: every partial sum is exact, so both paths agree bit for bit."""
    case = make_case(dtype, 1800, 7000, 2048, out="f32", dist="int")
    assert _split_last_wave(case, dgl.OUT_F32), "test setup: this shape should split its last wave"
    A, B, sa, sb = gu.to_device(case)
    ref, intact = _call(case, A, B, sa, sb, noalloc=False)
    assert intact
    for call in range(2):
        got, intact = _call(case, A, B, sa, sb, noalloc=True)
        assert intact
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), f"call {call}: differs"


def test_noalloc_decode_shape_runs_without_the_array():
    """m <= 16 takes the decode path, which needs no scratch; results match too."""
    case = make_case("bf16", 8, 4096, 4096, out="f32", dist="normal")
    A, B, sa, sb = gu.to_device(case)
    ref, _ = _call(case, A, B, sa, sb, noalloc=False)
    got, intact = _call(case, A, B, sa, sb, noalloc=True)
    assert intact
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))


def test_noalloc_allocates_no_device_memory():
    """The defining property: a call on a fresh stream leaves the device's free
    memory unchanged, where the stream-K path of dgl_gemm_planned allocates a
    workspace of at least 24 MiB for the same problem on a fresh stream."""
    case = make_case("bf16", 1800, 7000, 2048, out="f32", dist="normal")
    assert _split_last_wave(case, dgl.OUT_F32), "test setup: this shape should split its last wave"
    A, B, _sa, _sb = gu.to_device(case)
    C = torch.empty((case.m, case.n), dtype=torch.float32, device="cuda")
    s_warm, s_new, s_ctl = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def noalloc(stream):
        return dgl.dgl_gemm_noalloc(dgl.DTYPE_BF16, A.data_ptr(), B.data_ptr(), None, None, C.data_ptr(),
                                    case.m, case.n, case.K, case.m, case.n, dgl.OUT_F32, stream.cuda_stream)

    assert noalloc(s_warm) == dgl.DGL_OK  # first call: set-up, kernel modules loaded
    assert dgl.dgl_shutdown() == dgl.DGL_OK  # no workspace left from earlier tests
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    assert noalloc(s_new) == dgl.DGL_OK
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert dgl.dgl_device_status(s_new.cuda_stream) == dgl.DGL_OK
    assert free1 == free0, f"dgl_gemm_noalloc changed free device memory by {free0 - free1} bytes"
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, stream_k=1)
    st = dgl.dgl_gemm_planned(dgl.DTYPE_BF16, A.data_ptr(), B.data_ptr(), None, None, C.data_ptr(), case.m,
                              case.n, case.K, case.m, case.n, dgl.OUT_F32, plan, s_ctl.cuda_stream)
    assert st == dgl.DGL_OK
    torch.cuda.synchronize()
    free2 = torch.cuda.mem_get_info()[0]
    assert free1 - free2 >= 24 << 20, "control: the allocating path should have taken a workspace"
    assert dgl.dgl_shutdown() == dgl.DGL_OK
