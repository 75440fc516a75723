"""Every workload at full size, in the launch configuration the benchmark
times (the planner's choice), checked on a seeded sample of 4096 outputs plus
full tiles at every ragged edge, and guard-banded against stray writes."""
import pytest

import dense_gemm_linear_gb300 as dgl
from synthetic import FP8_SHAPES, LLAMA_SHAPES, RAGGED_SWEEP, SQUARE_SHAPES, make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _check(case, guard=True):
    Cbuf, intact = gu.run(case, guard_rows=2 if guard else 0, pad_cols=8 if guard else 0)
    assert intact, f"{case.name}: wrote outside the valid region"
    plan = dgl.dgl_plan(0 if case.dtype == "bf16" else 1, case.m, case.n, case.K,
                        dgl.OUT_F32 if case.out == "f32" else dgl.OUT_BF16)
    tm = plan.tile_m if plan.path == dgl.PATH_TC else 256
    tn = plan.tile_n if plan.path == dgl.PATH_TC else 256
    if case.m * case.n * case.K <= (1 << 30):
        gu.assert_close_full(case, gu.host_valid(case, Cbuf))
    else:
        gu.assert_close_sampled(case, Cbuf, tm, tn, seed=case.seed)


@pytest.mark.parametrize("m,n,k", RAGGED_SWEEP, ids=lambda v: str(v))
def test_ragged_sweep(m, n, k):
    _check(make_case("bf16", m, n, k, out="bf16"))


@pytest.mark.parametrize("m,n,k", RAGGED_SWEEP, ids=lambda v: str(v))
def test_ragged_sweep_tight_pitch(m, n, k):
    """C pitch = n: a stray column would land on the next row, where the product check sees it."""
    _check(make_case("bf16", m, n, k, out="bf16"), guard=False)


@pytest.mark.parametrize("m,n,k", LLAMA_SHAPES, ids=lambda v: str(v))
def test_llama7b_mlp(m, n, k):
    _check(make_case("bf16", m, n, k, out="bf16"))


@pytest.mark.parametrize("m,n,k", SQUARE_SHAPES, ids=lambda v: str(v))
def test_squares(m, n, k):
    _check(make_case("bf16", m, n, k, out="bf16", a_std=1.0, b_std=1.0))


@pytest.mark.parametrize("m,n,k", FP8_SHAPES, ids=lambda v: str(v))
def test_fp8(m, n, k):
    _check(make_case("fp8", m, n, k, out="bf16", dist="fp8"))


@pytest.mark.parametrize("m,n,k", [(4096, 4096, 4096), (597, 11008, 4096), (16, 11008, 4096)])
def test_fp8_integer_exact(m, n, k):
    """Integer E4M3 inputs with scales in {0.5, 1, 2}: fp32 output is exact (sampled)."""
    case = make_case("fp8", m, n, k, out="f32", dist="int")
    Cbuf, intact = gu.run(case)
    assert intact
    rows, cols = gu.sample_points(case, 256, 256, seed=1)
    import torch
    ref, _ = gu.oracle.gemm_points(gu.oracle.E4M3, case.A, case.B, rows, cols, case.sa, case.sb)
    got = Cbuf[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    assert (got == ref).all()
