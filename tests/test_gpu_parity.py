"""CUDA path vs the oracle, element by element, through the C ABI.

Small cases are compared in full; every case also checks that nothing outside
the valid region of C was written (guard rows and a padded row pitch filled
with NaN canaries, the guard-band idea of FlyDSL pull request 1303's tests).
Tolerances: |C - C_ref| <= 1e-4 * sum_k |a_ik b_jk| + 1e-6 for fp32 output,
plus 1e-2 |C_ref| for bf16 output; integer-valued inputs must match exactly.
"""
import numpy as np
import pytest

import dense_gemm_linear_gb300 as dgl
from synthetic import make_case
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _full(case, **kw):
    Cbuf, intact = gu.run(case, **kw)
    assert intact, f"{case.name}: wrote outside the valid region"
    C = gu.host_valid(case, Cbuf)
    gu.assert_close_full(case, C)
    return C


# -------------------------------------------------------------- the 256^3 case
def test_square256_uniform_f32():
    _full(make_case("bf16", 256, 256, 256, out="f32", dist="uniform"))


def test_square256_integer_bit_exact():
    case = make_case("bf16", 256, 256, 256, out="f32", dist="int")
    Cbuf, intact = gu.run(case)
    assert intact
    gu.assert_exact(case, gu.host_valid(case, Cbuf))


# -------------------------------------------------------------- structure pins on the GPU path
def test_identity_gives_transpose():
    """A = I_K: C = B^T exactly, so any layout mistake shows as a permutation."""
    K, n = 128, 192
    case = make_case("bf16", K, n, K, out="f32", dist="int")
    eye = np.eye(K)
    from synthetic import to_bf16_codes
    case.A = to_bf16_codes(eye)
    Cbuf, intact = gu.run(case)
    assert intact
    C = gu.host_valid(case, Cbuf)
    Bv = gu.oracle.decode_bf16(case.B)
    np.testing.assert_array_equal(C, Bv.T)


SMALL_RAGGED = [(130, 200, 72), (1, 37, 64), (17, 300, 136), (129, 257, 200), (255, 65, 8),
                (300, 513, 1000), (16, 64, 4096), (33, 1000, 48), (500, 129, 2056)]


@pytest.mark.parametrize("m,n,k", SMALL_RAGGED)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_small_ragged_bf16(m, n, k, out):
    _full(make_case("bf16", m, n, k, out=out), guard_rows=3, pad_cols=5)


@pytest.mark.parametrize("m,n,k", SMALL_RAGGED)
def test_small_ragged_e4m3(m, n, k):
    if k % 16:
        pytest.skip("E4M3 rows must be a multiple of 16 bytes")
    _full(make_case("fp8", m, n, k, out="bf16", dist="fp8"), guard_rows=2, pad_cols=3)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("m", [1, 5, 16, 40, 200])
def test_integer_bit_exact_all_paths(dtype, m):
    case = make_case(dtype, m, 300, 512, out="f32", dist="int")
    Cbuf, intact = gu.run(case, guard_rows=1, pad_cols=2)
    assert intact
    gu.assert_exact(case, gu.host_valid(case, Cbuf))


# -------------------------------------------------------------- every ladder rung, forced
LADDER = [(dgl.PATH_TC, 64, 64), (dgl.PATH_TC, 64, 128), (dgl.PATH_TC, 64, 256),
          (dgl.PATH_TC, 128, 64), (dgl.PATH_TC, 128, 128), (dgl.PATH_TC, 128, 256), (dgl.PATH_TC, 256, 128),
          (dgl.PATH_TC, 256, 224), (dgl.PATH_TC, 256, 256)]


@pytest.mark.parametrize("path,tm,tn", LADDER, ids=lambda v: str(v))
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_forced_tile_on_shape_no_tile_divides(path, tm, tn, dtype, out):
    """Each rung on a shape none of them divides (ragged in M, N and K)."""
    case = make_case(dtype, 333, 517, 336, out=out, dist="fp8" if dtype == "fp8" else "normal")
    plan = dgl.PlanInfo(path=path, tile_m=tm, tile_n=tn)
    _full(case, plan=plan, guard_rows=4, pad_cols=7)


@pytest.mark.parametrize("pad,base", [(0, 0), (8, 0), (3, 0), (1, 1), (0, 1), (5, 3)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("tm,tn", [(64, 64), (64, 256), (128, 64), (128, 128), (128, 256), (256, 128), (256, 224),
                                   (256, 256)])
def test_output_store_paths(pad, base, out, tm, tn):
    """C pitch and base alignment select the TMA-store or the predicated-store
    epilogue; odd pitches alternate row alignment, an odd base shifts every row."""
    case = make_case("bf16", 261, 328, 200, out=out)
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm, tile_n=tn)
    Cbuf, intact = gu.run(case, plan=plan, guard_rows=2, pad_cols=pad, base_offset=base)
    assert intact, "wrote outside the valid region"
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("n", [1, 2, 3, 5, 7, 8, 9, 15, 17, 23])
@pytest.mark.parametrize("base", [0, 1, 3])
@pytest.mark.parametrize("tm,tn", [(64, 64), (128, 256), (256, 256)])
def test_row_staging_rows_shorter_than_a_unit(n, base, tm, tn):
    """bf16 C rows of a few columns at a pitch or base that is not 16-byte
    aligned: a row's bytes fit in one or two partial 16-byte units (no aligned
    body), which the end-unit stores write alone."""
    case = make_case("bf16", 40, n, 64, out="bf16")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm, tile_n=tn)
    Cbuf, intact = gu.run(case, plan=plan, guard_rows=2, pad_cols=3, base_offset=base)
    assert intact, "wrote outside the valid region"
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("tm,grid", [(64, 1), (64, 5), (128, 1), (128, 3), (128, 7), (256, 2), (256, 6)])
def test_persistent_tile_loop_small_grid(tm, grid):
    """Fewer CTAs (or CTA pairs) than tiles: each walks many tiles through both accumulators."""
    case = make_case("bf16", 700, 900, 264, out="f32")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm, tile_n=128, grid=grid)
    _full(case, plan=plan)


@pytest.mark.parametrize("tm,tn", [(128, 128), (128, 256), (256, 128), (256, 224), (256, 256)])
@pytest.mark.parametrize("m,n,k", [(700, 900, 2048), (300, 520, 4096), (1030, 1000, 1024)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_stream_k_split_tiles(tm, tn, m, n, k, out):
    """Stream-K: tiles of the partial last wave split along K across workers,
    partials handed over through the workspace (guard bands on C)."""
    case = make_case("bf16", m, n, k, out=out)
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm, tile_n=tn, stream_k=1)
    _full(case, plan=plan, guard_rows=2, pad_cols=3)


@pytest.mark.parametrize("tm,tn", [(128, 256), (256, 256)])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_stream_k_integer_exact_and_repeatable(tm, tn, dtype):
    """Integer inputs: split sums are exact in fp32, so stream-K must match the
    exact result bit for bit, on back-to-back launches sharing the workspace."""
    case = make_case(dtype, 900, 1100, 2048, out="f32", dist="int")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm, tile_n=tn, stream_k=1)
    ops = gu.to_device(case)
    for _ in range(3):
        Cbuf, intact = gu.run(case, plan=plan, dev_ops=ops)
        assert intact
        gu.assert_exact(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("m", [1, 3, 8, 16])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 2049])
def test_decode_path(dtype, m, n):
    case = make_case(dtype, m, n, 256, out="bf16", dist="fp8" if dtype == "fp8" else "normal")
    assert dgl.dgl_plan(0 if dtype == "bf16" else 1, m, n, 256).path == dgl.PATH_DECODE
    _full(case, guard_rows=2, pad_cols=3)


@pytest.mark.parametrize("ks", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_decode_forced_stage_widths(ks, dtype):
    """Every decode stage width (128-byte K steps per ring stage), with a K tail
    that leaves the last stage partly filled."""
    k = 1040 if dtype == "bf16" else 2080
    case = make_case(dtype, 5, 777, k, out="f32", dist="fp8" if dtype == "fp8" else "normal")
    kstep = 64 if dtype == "bf16" else 128
    _full(case, plan=dgl.PlanInfo(path=dgl.PATH_DECODE, tile_k=ks * kstep), guard_rows=1, pad_cols=2)


@pytest.mark.parametrize("k", [16, 48, 272, 4104, 8192])
def test_decode_k_extents(k):
    _full(make_case("bf16", 7, 300, k, out="f32"))


def test_decode_many_rows_per_cta():
    """n large enough that each CTA reduces several 128-row blocks."""
    case = make_case("bf16", 4, 50257, 64, out="bf16")
    Cbuf, intact = gu.run(case, pad_cols=1)
    assert intact
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("m", list(range(1, 17)))
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_decode_every_m(m, out):
    """The decode path for every m in both output types; n = 1001 leaves
    ragged parts and K = 264 a partial 128-byte step."""
    _full(make_case("bf16", m, 1001, 264, out=out), guard_rows=1, pad_cols=3)


@pytest.mark.parametrize("m", list(range(1, 17)))
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_decode_every_m_whole_k_steps(m, dtype):
    """K a whole number of 128-byte steps: each stage's A planes arrive as one
    3-D box of 16 rows (zeros past m); every m, ragged parts, and a last
    stage with fewer K steps than the box (zeros past K)."""
    k = 640 if dtype == "bf16" else 1280   # ten 128-byte steps: stages of 8 and 2
    case = make_case(dtype, m, 1001, k, out="f32", dist="fp8" if dtype == "fp8" else "normal")
    _full(case, guard_rows=1, pad_cols=3)


@pytest.mark.parametrize("dtype,n,k,g", [("bf16", 1100, 1024, 16), ("bf16", 2000, 512, 8), ("bf16", 4000, 1024, 4),
                                         ("bf16", 9000, 512, 2), ("fp8", 1100, 2048, 16), ("fp8", 4000, 2048, 4)])
@pytest.mark.parametrize("m,out", [(1, "bf16"), (7, "f32"), (16, "bf16")])
def test_decode_stacked_k_steps(dtype, n, k, g, m, out):
    """Parts of at most 128 / G rows: G K steps share one MMA and the epilogue
    adds the G diagonal blocks (every G, ragged parts since 152 divides no n)."""
    assert dgl.dgl_plan(0 if dtype == "bf16" else 1, m, n, k).k_group == g
    case = make_case(dtype, m, n, k, out=out, dist="fp8" if dtype == "fp8" else "normal")
    _full(case, guard_rows=1, pad_cols=3)


@pytest.mark.parametrize("n,k,grid", [(2000, 512, 7), (1100, 1024, 3), (9000, 512, 64)])
def test_decode_stacked_many_parts_per_cta(n, k, grid):
    """A forced small grid: each CTA walks many parts, so the shared-memory
    partial sums and both TMEM buffers are reused; integer inputs, exact."""
    case = make_case("bf16", 9, n, k, out="f32", dist="int")
    Cbuf, intact = gu.run(case, plan=dgl.PlanInfo(path=dgl.PATH_DECODE, grid=grid), guard_rows=1, pad_cols=1)
    assert intact
    gu.assert_exact(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("m,n,k", [(1, 11008, 4096), (8, 4096, 4096), (16, 4096, 4096), (3, 16, 8)])
def test_decode_full_shapes(m, n, k):
    """The decode shapes of the benchmarks at full size (sampled), and K = 8."""
    case = make_case("bf16", m, n, k, out="f32")
    Cbuf, intact = gu.run(case, guard_rows=1, pad_cols=1)
    assert intact
    gu.assert_close_sampled(case, Cbuf, tile_m=16, tile_n=128)


def test_forced_decode_vs_tile_same_result():
    """m <= 16 through both paths: both within tolerance of the oracle."""
    case = make_case("bf16", 12, 640, 512, out="f32")
    _full(case, plan=dgl.PlanInfo(path=dgl.PATH_TC, tile_m=128, tile_n=128))
    _full(case, plan=dgl.PlanInfo(path=dgl.PATH_DECODE))


def test_deterministic_repeat():
    case = make_case("bf16", 600, 700, 1024, out="f32")
    ops = gu.to_device(case)
    a, _ = gu.run(case, dev_ops=ops)
    b, _ = gu.run(case, dev_ops=ops)
    assert bool((a == b).all().item())


# -------------------------------------------------------------- degenerate cases and errors
def test_k_zero_writes_zeros():
    import torch
    C = gu.canary_buffer(5, 9, "f32")
    A = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    st = dgl.dgl_gemm_bf16(A.data_ptr(), A.data_ptr(), C.data_ptr(), 5, 9, 0, 4, 7, dgl.OUT_F32, 0)
    assert st == dgl.DGL_OK
    torch.cuda.synchronize()
    c = C.cpu().numpy()
    assert (c[:4, :7] == 0).all()
    assert np.isnan(c[4, :]).all() and np.isnan(c[:, 7:]).all()


def test_empty_product_is_noop():
    assert dgl.dgl_gemm_bf16(None, None, None, 0, 10, 64, 0, 0, dgl.OUT_BF16, 0) == dgl.DGL_OK
    assert dgl.dgl_gemm_bf16(None, None, None, 10, 0, 64, 0, 0, dgl.OUT_BF16, 0) == dgl.DGL_OK


def test_argument_errors():
    import torch
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    p = A.data_ptr()
    assert dgl.dgl_gemm_bf16(p, p, C.data_ptr(), 64, 64, 60, 0, 0, 0, 0) == dgl.DGL_ERR_ALIGN  # K % 8
    assert dgl.dgl_gemm_bf16(p + 2, p, C.data_ptr(), 64, 64, 64, 0, 0, 0, 0) == dgl.DGL_ERR_ALIGN
    assert dgl.dgl_gemm_bf16(p, p, C.data_ptr(), 64, 64, 64, 65, 0, 0, 0) == dgl.DGL_ERR_ARG
    assert dgl.dgl_gemm_bf16(None, p, C.data_ptr(), 64, 64, 64, 0, 0, 0, 0) == dgl.DGL_ERR_ARG
    assert dgl.dgl_gemm_bf16(p, p, C.data_ptr(), 64, 64, 64, 0, 0, 7, 0) == dgl.DGL_ERR_ARG
    assert dgl.dgl_gemm_fp8(p, p, None, None, C.data_ptr(), 64, 64, 64, 0, 0, 0, 0) == dgl.DGL_ERR_ARG
    assert dgl.dgl_gemm_bf16(p, p, C.data_ptr(), 64, 64, 1 << 31, 0, 0, 0, 0) == dgl.DGL_ERR_SHAPE
    bad = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=128, tile_n=96)
    assert dgl.dgl_gemm_planned(0, p, p, None, None, C.data_ptr(), 64, 64, 64, 0, 0, 0, bad, 0) == \
        dgl.DGL_ERR_UNSUPPORTED
    assert dgl.dgl_device_status(0) == dgl.DGL_OK


def test_torch_helpers_and_streams():
    import torch
    case = make_case("bf16", 200, 300, 128, out="bf16")
    A, B, _, _ = gu.to_device(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = dgl.gemm_bf16(A, B)
    s.synchronize()
    gu.assert_close_full(case, C.double().cpu().numpy())


# -------------------------------------------------------------- split tail (half tiles in the last wave)
SPLIT_TAIL_CASES = [
    # (m, n, k, tile, dtype, out): at least one full wave, a tail of at most half the workers
    (2304, 2304, 256, (256, 256), "bf16", "bf16"),    # 81 pair tiles: 76 + a tail of 5
    (2300, 2290, 200, (256, 256), "bf16", "bf16"),    # ragged m, n, K; unaligned bf16 rows
    (2304, 2304, 256, (256, 256), "fp8", "bf16"),
    (1280, 4096, 128, (128, 256), "bf16", "f32"),      # 160 one-CTA tiles: 152 + a tail of 8
    (1290, 4000, 136, (128, 256), "bf16", "bf16"),
]


@pytest.mark.parametrize("m,n,k,tile,dtype,out", SPLIT_TAIL_CASES)
def test_split_tail(m, n, k, tile, dtype, out):
    case = make_case(dtype, m, n, k, out=out, dist="fp8" if dtype == "fp8" else "normal")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tile[0], tile_n=tile[1], split_tail=1)
    Cbuf, intact = gu.run(case, plan=plan, guard_rows=1, pad_cols=1)
    assert intact
    gu.assert_close_full(case, gu.host_valid(case, Cbuf))


def test_split_tail_integer_exact():
    case = make_case("bf16", 2304, 2304, 128, out="f32", dist="int")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=256, split_tail=1)
    Cbuf, intact = gu.run(case, plan=plan)
    assert intact
    gu.assert_exact(case, gu.host_valid(case, Cbuf))


# -------------------------------------------------------------- 64-row rungs (M = 64 MMAs)
@pytest.mark.parametrize("tn", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("m", [1, 15, 16, 17, 63, 64, 65, 130])
def test_m64_rungs_integer_exact(tn, dtype, m):
    """64-row tiles hold 16 rows per epilogue warp (tensor-memory lanes
    32 q .. 32 q + 15): every row count around the 16-row warp slices and the
    64-row tile must come out exact, guard bands intact."""
    case = make_case(dtype, m, 300, 512, out="f32", dist="int")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=64, tile_n=tn)
    Cbuf, intact = gu.run(case, plan=plan, guard_rows=3, pad_cols=2)
    assert intact
    gu.assert_exact(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("tn", [64, 128, 256])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_m64_rungs_long_k_many_tiles(tn, out):
    """Several waves of 64-row tiles through both accumulators, K of 4096."""
    case = make_case("bf16", 333, 1100, 4096, out=out)
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=64, tile_n=tn)
    _full(case, plan=plan, guard_rows=2, pad_cols=5)


def test_m64_rejected_for_mn_major_and_linear():
    """64-row tiles are plain K-major GEMMs: other forced uses are refused."""
    import torch
    case = make_case("bf16", 128, 128, 64, out="f32")
    A, B, _, _ = gu.to_device(case)
    C = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=64, tile_n=128)
    st = dgl.dgl_gemm_bf16_ex(dgl.MN_MAJOR, dgl.K_MAJOR, A.data_ptr(), 0, B.data_ptr(), 0, C.data_ptr(), 0, 128,
                              128, 64, dgl.OUT_F32, plan, torch.cuda.current_stream().cuda_stream)
    assert st == dgl.DGL_ERR_UNSUPPORTED
    st = dgl.dgl_linear(dgl.DTYPE_BF16, A.data_ptr(), B.data_ptr(), None, None, None, C.data_ptr(), 128, 128, 64,
                        128, 128, dgl.OUT_F32, dgl.ACT_GELU, 0, plan, torch.cuda.current_stream().cuda_stream)
    assert st == dgl.DGL_ERR_UNSUPPORTED


# -------------------------------------------------------------- split-K tail (stream_k = S >= 2)
# One whole wave plus a tail of 19 tiles: 76 CTA pairs (or 152 CTAs) leave room
# for up to four workers per tail tile.
SPLIT_K_SHAPES = {(256, 256): (1200, 4800), (256, 128): (1200, 2400), (128, 256): (1250, 4800)}


@pytest.mark.parametrize("tm,tn", list(SPLIT_K_SHAPES))
@pytest.mark.parametrize("ways", [2, 4])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_split_k_tail_integer_exact(tm, tn, ways, dtype):
    """Each tail tile's k-stages in `ways` tile-aligned ranges, partials added by
    the worker holding the first range: exact on integer inputs, twice in a
    row on the shared workspace."""
    m, n = SPLIT_K_SHAPES[(tm, tn)]
    case = make_case(dtype, m, n, 512, out="f32", dist="int")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm, tile_n=tn, stream_k=ways)
    ops = gu.to_device(case)
    for _ in range(2):
        Cbuf, intact = gu.run(case, plan=plan, dev_ops=ops, guard_rows=2, pad_cols=3)
        assert intact
        gu.assert_exact(case, gu.host_valid(case, Cbuf))


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_split_k_tail_general_values(out):
    """The planner's own choice for a long-K shape with a short tail (K = 4096,
    four workers per tail tile): a seeded sample and whole corner tiles."""
    case = make_case("bf16", 1200, 4800, 4096, out=out)
    p = dgl.dgl_plan(dgl.DTYPE_BF16, case.m, case.n, case.K, dgl.OUT_F32 if out == "f32" else dgl.OUT_BF16,
                     num_sms=152)
    assert p.stream_k >= 2, "test setup: the planner should split this tail"
    Cbuf, intact = gu.run(case, guard_rows=2, pad_cols=5)
    assert intact
    gu.assert_close_sampled(case, Cbuf, p.tile_m, p.tile_n)


# -------------------------------------------------------------- the 224-wide pair tile
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_pair_224_integer_exact_full_waves(dtype, out):
    """256 x 224 pair tiles: the accumulators sit 256 tensor-memory columns
    apart and a lane quarter's two warps take 4 + 3 of the 7 chunks.  Exact on
    integer inputs over several waves, with ragged edges and guard bands."""
    case = make_case(dtype, 1100, 3000, 512, out=out, dist="int")
    plan = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=256, tile_n=224)
    Cbuf, intact = gu.run(case, plan=plan, guard_rows=2, pad_cols=3)
    assert intact
    if out == "f32":
        gu.assert_exact(case, gu.host_valid(case, Cbuf))
    else:
        gu.assert_close_full(case, gu.host_valid(case, Cbuf))
