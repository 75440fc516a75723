"""Host-side checks that need no GPU: the C ABI library loads and exports
every symbol include/dgl.h declares; the planner's metric helpers match the
worked examples printed on the pages; planner rules; the input generator."""
import ctypes
import json
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dgl.h")


@pytest.fixture(scope="module")
def dgl():
    import dense_gemm_linear_gb300 as d
    from dense_gemm_linear_gb300 import _build
    _build.build()
    d.load_library()
    return d


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dgl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("dgl_gemm_bf16", "dgl_gemm_fp8", "dgl_gemm_planned", "dgl_plan", "dgl_tile_metrics",
                 "dgl_device_status", "dgl_status_string", "dgl_version"):
        assert must in names


def test_library_exports_every_declared_symbol(dgl):
    lib = ctypes.CDLL(dgl.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in dgl.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", dgl.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(dgl_[a-z0-9_]+)\b", out))
    assert set(declared_functions()) <= exported
    assert set(dgl.EXPORTED) == set(declared_functions())


def test_version_and_status_strings(dgl):
    assert dgl.dgl_version() >= 100
    for code in range(-6, 1):
        assert dgl.status_string(code) not in ("", "unknown status")


# ------------------------------------------------------------ TraceLens worked examples
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("idx", range(3))
def test_tile_metrics_tracelens_examples(dgl, idx):
    """The page's calculation examples and output row (tests/golden/tracelens_dim_eff.json):
    tile count, tile_eff, wq_eff and dim_eff to the digits the page prints."""
    g = _golden("tracelens_dim_eff.json")
    c = g["cases"][idx]
    m = dgl.dgl_tile_metrics(c["m"], c["n"], c["mt_m"], c["mt_n"], g["num_units"])
    assert m.num_tiles == c["num_tiles"]
    tol = 10.0 ** -c["digits"]  # the page rounds or truncates ("approximately") to these digits
    assert abs(m.wq_eff - c["wq_eff"]) <= tol and abs(m.dim_eff - c["dim_eff"]) <= tol
    assert abs(m.tile_eff - c["tile_eff"]) < 1e-4
    assert -(-m.num_tiles // g["num_units"]) == c["rounds"]


def test_tile_metrics_errors(dgl):
    with pytest.raises(dgl.DglError):
        dgl.dgl_tile_metrics(10, 10, 0, 64, 10)
    with pytest.raises(dgl.DglError):
        dgl.dgl_tile_metrics(10, 10, 64, 64, 0)


# ------------------------------------------------------------ the guide's worked example
def test_guide_worked_example_flops_and_bytes():
    """tests/golden/gemm_guide_worked_example.json: 436 GFLOP and 137.6 MB; at
    ~500 TFLOP/s that is ~0.87 ms and ~158 GB/s."""
    from dense_gemm_linear_gb300 import metrics
    g = _golden("gemm_guide_worked_example.json")
    f = metrics.gemm_flops(g["m"], g["n"], g["k"])
    b = metrics.gemm_bytes(g["m"], g["n"], g["k"], in_bytes=g["in_bytes"], out_bytes=g["out_bytes"],
                           scaled=g["scaled"])
    assert round(f / 1e9) == g["gflop"]
    assert abs(b / 1e6 - g["mbytes"]) < 0.1          # 137.67 MB; the page truncates to 137.6
    t = f / (g["target_tflops"] * 1e12)
    assert round(t * 1e3, 2) == g["ms"]
    assert round(b / t / 1e9) == g["gbs"]


def test_arithmetic_intensity_classification():
    from dense_gemm_linear_gb300 import metrics
    # decode is memory-bound, large squares compute-bound, on GB300's ~281 flop/byte crossover
    assert metrics.arithmetic_intensity(1, 11008, 4096) < 2
    assert metrics.arithmetic_intensity(4096, 4096, 4096) > 1000


# ------------------------------------------------------------ planner rules
def test_plan_decode_threshold(dgl):
    for m in (1, 4, 16):
        assert dgl.dgl_plan(0, m, 11008, 4096, num_sms=152).path == dgl.PATH_DECODE
    assert dgl.dgl_plan(0, 17, 11008, 4096, num_sms=152).path == dgl.PATH_TC
    assert dgl.dgl_plan(0, 0, 10, 10, num_sms=152).path == dgl.PATH_EMPTY


@pytest.mark.parametrize("dtype,n,k,want", [(0, 11008, 4096, 1), (0, 4096, 4096, 4), (0, 1100, 1024, 16),
                                             (0, 2000, 512, 8), (0, 9000, 512, 2), (0, 1001, 264, 1),
                                             (0, 300, 8192, 16), (0, 300, 4104, 1), (1, 4000, 2048, 4),
                                             (1, 11008, 4096, 1), (0, 50257, 64, 1)])
def test_plan_decode_k_group(dgl, dtype, n, k, want):
    """Decode parts of at most 128 / G rows stack G 128-byte K steps into one
    128-row MMA operand: G is the largest power of two <= 16 whose slots hold
    the part and that divides the step count; each ring stage is whole groups."""
    p = dgl.dgl_plan(dtype, 8, n, k, num_sms=152)
    assert p.path == dgl.PATH_DECODE
    assert p.k_group == want
    nk = -(-k * (1 if dtype == 1 else 2) // 128)
    g = p.k_group
    assert p.tile_n <= 128 // g and nk % g == 0
    assert g == 16 or p.tile_n > 128 // (2 * g) or nk % (2 * g) != 0
    ks = p.tile_k // (128 if dtype == 1 else 64)
    assert ks % g == 0 and p.stages >= 2
    assert dgl.dgl_plan(0, 600, 600, 600, num_sms=152).k_group == 1


@pytest.mark.parametrize("dtype,m,n,k,tile", [(0, 1024, 50257, 512, (128, 256)), (0, 2048, 2048, 2048, (128, 256)),
                                              (0, 48, 4096, 48, (64, 64)), (0, 528, 528, 1024, (64, 64)),
                                              (0, 3402, 4096, 1024, (256, 256)), (0, 597, 11008, 4096, (256, 256)),
                                              (1, 597, 11008, 4096, (256, 256))])
def test_plan_measured_pins(dgl, dtype, m, n, k, tile):
    """Shapes whose best tile was measured on GB300 take that tile."""
    p = dgl.dgl_plan(dtype, m, n, k, num_sms=152)
    assert p.path == dgl.PATH_TC and (p.tile_m, p.tile_n) == tile
    assert p.cta_group == (2 if tile[0] == 256 else 1)


def test_plan_decode_invariants_sweep(dgl):
    """Over a seeded sweep of n and K: parts of at most 128 / G rows, G a power
    of two dividing the 128-byte K steps, whole groups per ring stage, and the
    ring within its 192 KB with at least two stages."""
    import numpy as np
    rng = np.random.default_rng(11)
    for _ in range(400):
        dtype = int(rng.integers(0, 2))
        n = int(rng.integers(1, 60000))
        K = int(rng.integers(1, 1200)) * 16
        p = dgl.dgl_plan(dtype, int(rng.integers(1, 17)), n, K, num_sms=152)
        assert p.path == dgl.PATH_DECODE
        g = p.k_group
        assert g in (1, 2, 4, 8, 16)
        nk = -(-K * (1 if dtype == 1 else 2) // 128)
        assert nk % g == 0
        assert p.tile_n <= 128 // g
        parts = p.num_tiles
        assert 1 <= parts <= n and p.tile_n == -(-n // parts)  # balanced parts of at most ceil(n / parts) rows
        ks = p.tile_k // (128 if dtype == 1 else 64)
        assert ks >= 1 and ks % g == 0 and ks <= max(nk, 1)
        slot_rows = 128 // g if g > 1 else -(-p.tile_n // 8) * 8
        assert p.stages >= 2 and p.stages * ks * (2048 + slot_rows * 128) <= 196608


@pytest.mark.parametrize("m,n,k", [(48, 4096, 48), (333, 4096, 1024), (528, 528, 1024), (3402, 4096, 1024),
                                   (1024, 50257, 512), (2048, 11007, 1024), (4095, 4095, 1024),
                                   (597, 11008, 4096), (4096, 4096, 4096), (8192, 8192, 8192), (17, 5, 64)])
def test_plan_padding_screen(dgl, m, n, k):
    """The chosen tile pads the output by at most 1.25x, unless no ladder tile
    can or a measured pin overrides the screen (the 597-token prefill, 528^2)."""
    p = dgl.dgl_plan(0, m, n, k, num_sms=152)
    pinned_past_screen = {(597, 11008, 4096), (528, 528, 1024)}
    assert p.path == dgl.PATH_TC
    padded = -(-m // p.tile_m) * p.tile_m * -(-n // p.tile_n) * p.tile_n
    nk = -(-k * 2 // 128)
    rungs = [(64, 64), (64, 128), (64, 256), (128, 64), (128, 128), (128, 256), (256, 128), (256, 256)]
    if nk <= 16:
        rungs.append((256, 224))
    any_ok = any(-(-m // tm) * tm * -(-n // tn) * tn <= 1.25 * m * n for tm, tn in rungs)
    if any_ok and (m, n, k) not in pinned_past_screen:
        assert padded <= 1.25 * m * n
    cg = 2 if p.tile_m == 256 else 1
    assert p.cta_group == cg
    assert p.grid == min(p.num_tiles, 152 // cg) * cg
    assert 0 < p.dim_eff <= 1.0 and p.est_us > 0


def test_plan_split_tail_rule(dgl):
    """The last partial wave of 256x256 pair tiles splits into half tiles only
    with at least one full wave before it, a tail of at most half the 76 pair
    workers, and K of at most 16 k-blocks of 128 bytes."""
    def plan(dt, m, n, k):
        p = dgl.dgl_plan(dt, m, n, k, num_sms=152)
        return (p.tile_m, p.tile_n, p.num_tiles, p.split_tail)

    # 336 tiles = 4 waves of 76 + 32: short K splits in both dtypes, long K does not
    assert plan(0, 2048, 10752, 1024) == (256, 256, 336, 1)
    assert plan(1, 2048, 10752, 2048) == (256, 256, 336, 1)
    assert plan(0, 2048, 10752, 2048) == (256, 256, 336, 0)
    assert plan(0, 2048, 10752, 4096) == (256, 256, 336, 0)
    # 344 tiles = 4 waves + 40: more than half the workers, no split
    assert plan(0, 2048, 11007, 1024) == (256, 256, 344, 0)
    # no full wave before the tail
    assert plan(0, 2048, 2048, 1024)[3] == 0


def test_plan_argument_errors(dgl):
    info = dgl.PlanInfo()
    lib = dgl.load_library()
    assert lib.dgl_plan(0, -1, 10, 10, 0, 152, ctypes.byref(info)) == dgl.DGL_ERR_ARG
    assert lib.dgl_plan(5, 10, 10, 10, 0, 152, ctypes.byref(info)) == dgl.DGL_ERR_ARG
    assert lib.dgl_plan(0, 10, 10, 10, 9, 152, ctypes.byref(info)) == dgl.DGL_ERR_ARG
    assert lib.dgl_plan(0, 1 << 31, 10, 10, 0, 152, ctypes.byref(info)) == dgl.DGL_ERR_SHAPE
    assert lib.dgl_plan(0, 10, 10, 10, 0, 152, None) == dgl.DGL_ERR_ARG


def test_gemm_rejects_bad_arguments_before_any_device_call(dgl):
    """Argument checks run before the library touches the GPU, so they work here."""
    lib = dgl.load_library()
    assert lib.dgl_gemm_bf16(16, 16, 16, 64, 64, 60, 0, 0, 0, None) == dgl.DGL_ERR_ALIGN      # K % 8
    assert lib.dgl_gemm_bf16(18, 16, 16, 64, 64, 64, 0, 0, 0, None) == dgl.DGL_ERR_ALIGN      # A not 16 B aligned
    assert lib.dgl_gemm_bf16(16, 16, 16, 64, 64, 64, 65, 0, 0, None) == dgl.DGL_ERR_ARG       # m_valid > M
    assert lib.dgl_gemm_bf16(None, 16, 16, 64, 64, 64, 0, 0, 0, None) == dgl.DGL_ERR_ARG
    assert lib.dgl_gemm_bf16(16, 16, 16, 64, 64, 64, 0, 0, 3, None) == dgl.DGL_ERR_ARG        # bad out dtype
    assert lib.dgl_gemm_fp8(16, 16, None, None, 16, 64, 64, 64, 0, 0, 0, None) == dgl.DGL_ERR_ARG
    assert lib.dgl_gemm_bf16(16, 16, 16, 64, 64, 1 << 31, 0, 0, 0, None) == dgl.DGL_ERR_SHAPE
    assert lib.dgl_gemm_bf16(None, None, None, 0, 64, 64, 0, 0, 0, None) == dgl.DGL_OK        # empty
    assert lib.dgl_gemm_planned(0, 16, 16, None, None, 16, 64, 64, 64, 0, 0, 0, None, None) == dgl.DGL_ERR_ARG


# ------------------------------------------------------------ synthetic inputs
def test_generator_is_counter_based():
    from synthetic import STREAM_A, normal, splitmix64_stream, uniform
    full = splitmix64_stream(0, STREAM_A, 0, 1000)
    part = splitmix64_stream(0, STREAM_A, 400, 100)
    assert np.array_equal(full[400:500], part)
    a = uniform(3, 1, (5000,), -1, 1)
    b = uniform(3, 1, (5000,), -1, 1)
    assert np.array_equal(a, b) and a.min() >= -1 and a.max() < 1
    x = normal(0, 0, (200000,))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_generator_known_splitmix64_values():
    """SplitMix64 with state s: the first output for state 0 after one increment is
    0xE220A8397B1DCDAF (the published reference sequence for seed 0)."""
    from synthetic.rng import _GOLDEN, _mix64
    z = np.array([0], dtype=np.uint64) + _GOLDEN
    assert int(_mix64(z)[0]) == 0xE220A8397B1DCDAF


def test_workload_shapes_and_encodings():
    from synthetic import make_case
    c = make_case("bf16", 3, 5, 8)
    assert c.A.dtype == np.uint16 and c.A.shape == (3, 8) and c.B.shape == (5, 8)
    c8 = make_case("fp8", 3, 5, 16, dist="fp8")
    assert c8.A.dtype == np.uint8 and c8.sa.shape == (3,) and c8.sb.shape == (5,)
    assert ((c8.sa >= 0.5) & (c8.sa < 2)).all()
    ci = make_case("fp8", 4, 4, 16, dist="int")
    assert set(np.unique(ci.sa)) <= {0.5, 1.0, 2.0}


def test_batch_descriptor_layout_matches_the_header(tmp_path):
    """The ctypes GemmDesc has the C struct dgl_gemm_desc's size and field offsets."""
    import dense_gemm_linear_gb300 as dgl_mod
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    fields = [f for f, _ in dgl_mod.GemmDesc._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stddef.h>\n#include <stdio.h>\n#include \"dgl.h\"\nint main(void) {\n"
                   "  printf(\"%zu\\n\", sizeof(dgl_gemm_desc));\n" +
                   "".join(f"  printf(\"%zu\\n\", offsetof(dgl_gemm_desc, {f}));\n" for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(dgl_mod.GemmDesc)] + [getattr(dgl_mod.GemmDesc, f).offset for f in fields]
    assert got == want


def test_batch_checks_every_item_before_any_device_call(dgl):
    """dgl_gemm_batch validates all items first: a bad item anywhere returns its
    status with nothing enqueued (no device is touched here), and a batch of
    empty items is a no-op."""
    ok = dict(dtype=dgl.DTYPE_BF16, out_dtype=dgl.OUT_BF16, A=16, B=16, C=16, M=64, N=64, K=64)
    lib = dgl.load_library()
    assert dgl.dgl_gemm_batch([ok, dict(ok, K=60)]) == dgl.DGL_ERR_ALIGN          # K * 2 bytes not a multiple of 16
    assert dgl.dgl_gemm_batch([dict(ok, dtype=9), ok]) == dgl.DGL_ERR_ARG
    assert dgl.dgl_gemm_batch([ok, dict(ok, m_valid=65)]) == dgl.DGL_ERR_ARG       # m_valid > M
    assert dgl.dgl_gemm_batch([dict(ok, dtype=dgl.DTYPE_E4M3)]) == dgl.DGL_ERR_ARG  # E4M3 without scales
    assert dgl.dgl_gemm_batch([dict(ok, dtype=dgl.DTYPE_MXFP4, K=48)]) == dgl.DGL_ERR_ALIGN   # K % 32
    assert dgl.dgl_gemm_batch([dict(ok, M=0), dict(ok, N=0)]) == dgl.DGL_OK
    assert dgl.dgl_gemm_batch([]) == dgl.DGL_OK
    assert lib.dgl_gemm_batch(None, 2, None) == dgl.DGL_ERR_ARG
    assert lib.dgl_gemm_batch(None, -1, None) == dgl.DGL_ERR_ARG
