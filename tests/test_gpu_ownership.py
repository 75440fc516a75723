"""The library's own device memory: the stream-K workspaces, how many of them
it keeps, and dgl_shutdown(), which releases them.

The caller owns every operand and output; the one allocation the library makes
is the fp32 partial-tile workspace of a stream-K plan, one per (device, stream).
These tests check that at most four are kept per device, that dgl_shutdown()
frees them, and that calls after a shutdown rebuild their state and still
match the oracle.
"""
import pytest
import torch

import dense_gemm_linear_gb300 as dgl
from synthetic import make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MIB = 1 << 20
WS_MIB = 26  # one workspace: 24 MiB of partial tiles, its flags, rounded up to 2 MiB pages


def _stream_k_call(case, ops, C, stream):
    A, B, sa, sb = ops
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, stream_k=1)
    out_dtype = dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16
    st = dgl.dgl_gemm_planned(dgl.DTYPE_BF16, A.data_ptr(), B.data_ptr(), None, None, C.data_ptr(), case.m, case.n,
                              case.K, case.m, case.n, out_dtype, plan, stream.cuda_stream)
    assert st == dgl.DGL_OK, dgl.status_string(st)


def _free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def test_shutdown_frees_workspace_and_calls_rebuild():
    case = make_case("bf16", 700, 900, 2048, out="f32")
    ops = gu.to_device(case)
    C = torch.empty((case.m, case.n), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    _stream_k_call(case, ops, C, s)
    s.synchronize()
    assert dgl.dgl_device_status(s.cuda_stream) == dgl.DGL_OK
    gu.assert_close_full(case, C.double().cpu().numpy())
    before = _free_bytes()
    assert dgl.dgl_shutdown() == dgl.DGL_OK
    after = _free_bytes()
    assert after - before >= 24 * MIB, f"shutdown freed only {(after - before) / MIB:.1f} MiB"
    C.fill_(float("nan"))
    _stream_k_call(case, ops, C, s)
    s.synchronize()
    assert dgl.dgl_device_status(s.cuda_stream) == dgl.DGL_OK
    gu.assert_close_full(case, C.double().cpu().numpy())
    assert dgl.dgl_shutdown() == dgl.DGL_OK


def test_shutdown_twice_and_without_workspaces_is_ok():
    assert dgl.dgl_shutdown() == dgl.DGL_OK
    assert dgl.dgl_shutdown() == dgl.DGL_OK
    case = make_case("bf16", 200, 333, 136, out="bf16")
    Cbuf, intact = gu.run(case)
    assert intact
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


def test_workspaces_per_device_are_bounded():
    """Six streams each run a stream-K plan; at most four workspaces stay."""
    case = make_case("bf16", 700, 900, 2048, out="f32")
    ops = gu.to_device(case)
    streams = [torch.cuda.Stream() for _ in range(6)]
    outs = [torch.empty((case.m, case.n), dtype=torch.float32, device="cuda") for _ in streams]
    assert dgl.dgl_shutdown() == dgl.DGL_OK
    before = _free_bytes()
    for s, C in zip(streams, outs):
        _stream_k_call(case, ops, C, s)
    used = (before - _free_bytes()) / MIB
    assert 24 <= used <= 4 * WS_MIB + 4, f"{used:.1f} MiB held after six streams"
    first = None
    for s, C in zip(streams, outs):
        assert dgl.dgl_device_status(s.cuda_stream) == dgl.DGL_OK
        if first is None:
            first = C
            gu.assert_close_full(case, C.double().cpu().numpy())
        else:  # the same plan on the same data: the split sums add in the same order
            assert torch.equal(C.view(torch.int32), first.view(torch.int32))
    assert dgl.dgl_shutdown() == dgl.DGL_OK


def _graph_of(body, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body()
    return g


@pytest.mark.parametrize("warm", [True, False])
def test_split_schedule_in_a_cuda_graph(warm):
    """A split-K-tail plan captured in a CUDA graph and replayed three times
    gives the exact result every time: the launch leaves its flags cleared, so
    a replay (same parameters) cannot mistake old partials for new ones.  On
    a stream with no workspace yet (warm=False) the captured call allocates
    nothing and runs data-parallel."""
    case = make_case("bf16", 1200, 4800, 1024, out="f32", dist="int")
    A, B, _, _ = gu.to_device(case)
    C = torch.empty((case.m, case.n), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, stream_k=2)

    def call():
        st = dgl.dgl_gemm_planned(dgl.DTYPE_BF16, A.data_ptr(), B.data_ptr(), None, None, C.data_ptr(), case.m,
                                  case.n, case.K, case.m, case.n, dgl.OUT_F32, plan,
                                  torch.cuda.current_stream().cuda_stream)
        assert st == dgl.DGL_OK, dgl.status_string(st)

    assert dgl.dgl_shutdown() == dgl.DGL_OK
    if warm:
        with torch.cuda.stream(s):
            call()
        s.synchronize()
    before = _free_bytes()
    g = _graph_of(call, s)
    assert _free_bytes() >= before - 2 * MIB, "capture allocated a workspace"
    for _ in range(3):
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert dgl.dgl_device_status(0) == dgl.DGL_OK
        gu.assert_exact(case, C.double().cpu().numpy())
    del g
    assert dgl.dgl_shutdown() == dgl.DGL_OK
