"""The GEMM workloads, as seeded synthetic operands.

Shapes and value distributions follow the linear-layer GEMMs the pages work
with: the ragged-shape set of the FlyDSL RDNA3 pull request (decode batches of
1/8/16 tokens, 48 tokens against K=48, 3402-token prefill, the 1024x50257x512
lm_head, 2048x11007x1024, 4095^2x1024, 528^2x1024), the LLaMA-2-7B MLP up/gate
projection shapes of "GEMM analysis in TraceLens" (section "Real-world
example: LLaMA-2 7B": d_model 4096, d_ff 11008, prefill L=597, decode L=1),
large squares for peak throughput, and an fp8 (E4M3) set with per-row scales
on A and per-column scales on B.  No trained weights or datasets are involved:
activations are N(0,1) and weights N(0, 0.02^2) draws.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .encode import mx_quantize, pack_e2m1, to_bf16_codes, to_e2m1_codes, to_e4m3_codes
from .rng import STREAM_A, STREAM_B, STREAM_SA, STREAM_SB, integers, normal, uniform

# (m, n, K)
SMALL_SQUARE = [(256, 256, 256)]
RAGGED_SWEEP = [(1, 11008, 4096), (8, 4096, 4096), (16, 4096, 4096), (48, 4096, 48),
                (333, 4096, 1024), (528, 528, 1024), (3402, 4096, 1024), (1024, 50257, 512),
                (2048, 11007, 1024), (4095, 4095, 1024)]
LLAMA_SHAPES = [(597, 11008, 4096), (1, 11008, 4096), (4, 11008, 4096), (16, 11008, 4096)]
SQUARE_SHAPES = [(2048, 2048, 2048), (4096, 4096, 4096), (8192, 8192, 8192)]
FP8_SHAPES = [(4096, 4096, 4096), (597, 11008, 4096), (16, 11008, 4096)]
STREAM_BIAS = 4
ACT_IDS = {"none": 0, "gelu": 1, "silu": 2}


@dataclass
class GemmCase:
    """One GEMM problem: codes of A [m,K] and B [n,K], optional scales.

    dtype "mxfp4": A [m, K/2] and B [n, K/2] hold packed E2M1 codes and sa
    [m, K/32], sb [n, K/32] their E8M0 block-scale codes (uint8).
    dtype "w4a8": A [m, K] E4M3 codes, B [n, K/2] packed E2M1 codes, sa [m] and
    sb [n] fp32 scales."""
    dtype: str               # "bf16", "fp8", "mxfp4" or "w4a8"
    m: int
    n: int
    K: int
    out: str                 # "bf16" or "f32"
    dist: str                # recipe name
    seed: int
    A: np.ndarray = field(repr=False)   # uint16 (bf16 bits) or uint8 (E4M3 bits)
    B: np.ndarray = field(repr=False)
    sa: np.ndarray | None = field(default=None, repr=False)
    sb: np.ndarray | None = field(default=None, repr=False)
    # linear-layer epilogue (parameters only): activation 0 none / 1 GELU /
    # 2 SiLU, a bias per row of B, and gated = B holds 2n rows (gate, then up)
    act: int = 0
    gated: bool = False
    bias: np.ndarray | None = field(default=None, repr=False)
    # operand storage on the device: 0 K-major (A [m][K], B [n][K]), 1 MN-major
    # (A [K][m], B [K][n]); the codes above are always held K-major
    a_major: int = 0
    b_major: int = 0

    @property
    def name(self) -> str:
        return f"{self.dtype}_{self.m}x{self.n}x{self.K}_{self.dist}_{self.out}"

    @property
    def b_rows(self) -> int:
        return 2 * self.n if self.gated else self.n

    @property
    def linear(self) -> bool:
        return self.act != 0 or self.gated or self.bias is not None

    @property
    def flops(self) -> int:
        return 2 * self.m * self.b_rows * self.K


def make_case(dtype: str, m: int, n: int, K: int, *, out: str = "bf16",
              dist: str = "normal", seed: int = 0,
              a_std: float = 1.0, b_std: float = 0.02) -> GemmCase:
    """Build one case.

    dist:
      "normal"   A ~ N(0, a_std^2), B ~ N(0, b_std^2)            (bf16)
      "uniform"  A, B ~ U[-1, 1)                                 (bf16)
      "int"      A, B integers in [-4, 4]; fp8 scales in {0.5, 1, 2}
      "fp8"      x ~ N(0,1); sa, sb ~ U[0.5, 2); codes = e4m3(x / scale)
    dtype "mxfp4" (K a multiple of 32):
      "mx"       A ~ N(0, a_std^2), B ~ N(0, b_std^2), block-quantised (OCP MX)
      "int"      E2M1 codes of magnitude <= 3 with random signs, scale codes in
                 {126, 127, 128}: every product is a multiple of 2^-4 and sums
                 up to K = 4096 are exact in fp32
    """
    if dtype == "mxfp4":
        return _make_mx_case(m, n, K, out, dist, seed, a_std, b_std)
    if dtype == "w4a8":
        return _make_w4a8_case(m, n, K, out, dist, seed, b_std)
    if dtype not in ("bf16", "fp8"):
        raise ValueError(dtype)
    sa = sb = None
    if dist == "normal":
        a = normal(seed, STREAM_A, (m, K), 0.0, a_std)
        b = normal(seed, STREAM_B, (n, K), 0.0, b_std)
    elif dist == "uniform":
        a = uniform(seed, STREAM_A, (m, K), -1.0, 1.0)
        b = uniform(seed, STREAM_B, (n, K), -1.0, 1.0)
    elif dist == "int":
        a = integers(seed, STREAM_A, (m, K), -4, 4)
        b = integers(seed, STREAM_B, (n, K), -4, 4)
        if dtype == "fp8":
            pick = np.array([0.5, 1.0, 2.0], dtype=np.float32)
            sa = pick[integers(seed, STREAM_SA, (m,), 0, 2).astype(np.int64)]
            sb = pick[integers(seed, STREAM_SB, (n,), 0, 2).astype(np.int64)]
    elif dist == "fp8":
        if dtype != "fp8":
            raise ValueError("the fp8 recipe makes E4M3 codes")
        sa = uniform(seed, STREAM_SA, (m,), 0.5, 2.0).astype(np.float32)
        sb = uniform(seed, STREAM_SB, (n,), 0.5, 2.0).astype(np.float32)
        a = normal(seed, STREAM_A, (m, K)) / sa[:, None].astype(np.float64)
        b = normal(seed, STREAM_B, (n, K)) / sb[:, None].astype(np.float64)
    else:
        raise ValueError(dist)
    if dtype == "bf16":
        A, B = to_bf16_codes(a), to_bf16_codes(b)
    else:
        A, B = to_e4m3_codes(a), to_e4m3_codes(b)
        if sa is None:
            sa = np.ones(m, dtype=np.float32)
            sb = np.ones(n, dtype=np.float32)
    return GemmCase(dtype, m, n, K, out, dist, seed, A, B, sa, sb)


def _make_mx_case(m, n, K, out, dist, seed, a_std, b_std) -> GemmCase:
    if K % 32 != 0:
        raise ValueError("MXFP4 blocks: K must be a multiple of 32")
    if dist == "mx":
        A, sa = mx_quantize(normal(seed, STREAM_A, (m, K), 0.0, a_std))
        B, sb = mx_quantize(normal(seed, STREAM_B, (n, K), 0.0, b_std))
    elif dist == "int":
        codes = np.array([0, 1, 2, 3, 4, 5, 8, 9, 10, 11, 12, 13], dtype=np.uint8)  # |value| <= 3
        A = pack_e2m1(codes[integers(seed, STREAM_A, (m, K), 0, 11).astype(np.int64)])
        B = pack_e2m1(codes[integers(seed, STREAM_B, (n, K), 0, 11).astype(np.int64)])
        sa = (126 + integers(seed, STREAM_SA, (m, K // 32), 0, 2)).astype(np.uint8)
        sb = (126 + integers(seed, STREAM_SB, (n, K // 32), 0, 2)).astype(np.uint8)
    else:
        raise ValueError(dist)
    return GemmCase("mxfp4", m, n, K, out, dist, seed, A, B, sa, sb)


def _make_w4a8_case(m, n, K, out, dist, seed, b_std) -> GemmCase:
    """E4M3 activations and packed E2M1 weights (K even).

    "w4a8": activations x ~ N(0,1), sa ~ U[0.5, 2), codes e4m3(x / sa) (the
            fp8 recipe); weights w ~ N(0, b_std^2) with one scale per row,
            sb = max |w_row| / 6 (the row's largest magnitude on E2M1's
            largest value, 6), codes e2m1(w / sb), nearest, ties to even
    "int":  A integers in [-4, 4], B any E2M1 code (multiples of 1/2 up to 6),
            scales in {0.5, 1, 2}: every partial sum is a multiple of 1/4
            below 2^24, exact in fp32
    """
    if K % 2:
        raise ValueError("packed E2M1 rows: K must be even")
    if dist == "w4a8":
        sa = uniform(seed, STREAM_SA, (m,), 0.5, 2.0).astype(np.float32)
        A = to_e4m3_codes(normal(seed, STREAM_A, (m, K)) / sa[:, None].astype(np.float64))
        w = normal(seed, STREAM_B, (n, K), 0.0, b_std)
        amax = np.abs(w).max(axis=1)
        sb = np.where(amax > 0, amax / 6.0, 1.0).astype(np.float32)
        B = pack_e2m1(to_e2m1_codes(w / sb[:, None].astype(np.float64)))
    elif dist == "int":
        A = to_e4m3_codes(integers(seed, STREAM_A, (m, K), -4, 4))
        B = pack_e2m1(integers(seed, STREAM_B, (n, K), 0, 15).astype(np.uint8))
        pick = np.array([0.5, 1.0, 2.0], dtype=np.float32)
        sa = pick[integers(seed, STREAM_SA, (m,), 0, 2).astype(np.int64)]
        sb = pick[integers(seed, STREAM_SB, (n,), 0, 2).astype(np.int64)]
    else:
        raise ValueError(dist)
    return GemmCase("w4a8", m, n, K, out, dist, seed, A, B, sa, sb)


# name -> list of (dtype, m, n, K, out, dist)
WORKLOADS = {
    "square256": [("bf16", 256, 256, 256, "f32", "uniform"), ("bf16", 256, 256, 256, "f32", "int")],
    "ragged": [("bf16", m, n, k, "bf16", "normal") for (m, n, k) in RAGGED_SWEEP],
    "llama7b_mlp": [("bf16", m, n, k, "bf16", "normal") for (m, n, k) in LLAMA_SHAPES],
    "square": [("bf16", m, n, k, "bf16", "square_normal") for (m, n, k) in SQUARE_SHAPES],
    "fp8": [("fp8", m, n, k, "bf16", "fp8") for (m, n, k) in FP8_SHAPES],
    # linear layers with their epilogue: the GPT-3-XL forward addmm (TraceLens
    # "Real-world example: GPT-3-XL": 10240 x 8192 x 2048, bias) followed by
    # GELU, and the LLaMA-2 7B prefill up/gate pair as one gated call
    # one training step of a GPT-3-XL feed-forward projection (TraceLens
    # "Real-world example: GPT-3-XL", d_model 2048, d_ff 8192, 5 x 2048
    # tokens): the forward addmm with its bias and GELU, then dX = dY W
    # (B MN-major) and dW = dY^T X (both MN-major)
    "gpt3xl_train": [("bf16", 10240, 8192, 2048, "bf16", "normal", {"act": "gelu", "bias": True}),
                     ("bf16", 10240, 2048, 8192, "bf16", "normal", {"layout": ("k", "mn")}),
                     ("bf16", 8192, 2048, 10240, "bf16", "normal", {"layout": ("mn", "mn")})],
    # block-scaled FP4 (MXFP4; the GEMM guide's section 8.2 byte formula):
    # the square and the LLaMA-2 7B up/gate prefill and decode shapes, OCP MX
    # quantised N(0,1) activations and N(0, 0.02^2) weights
    "mxfp4": [("mxfp4", 4096, 4096, 4096, "bf16", "mx"), ("mxfp4", 597, 11008, 4096, "bf16", "mx"),
              ("mxfp4", 16, 11008, 4096, "bf16", "mx")],
    # 8-bit activations, 4-bit weights (the GEMM guide's section 8.2 formula
    # for 4-bit weights): the LLaMA-2 7B up/gate prefill and decode shapes and
    # the square, E4M3 activations and per-row-scaled E2M1 weights
    "w4a8": [("w4a8", 4096, 4096, 4096, "bf16", "w4a8"), ("w4a8", 597, 11008, 4096, "bf16", "w4a8"),
             ("w4a8", 16, 11008, 4096, "bf16", "w4a8"), ("w4a8", 1, 11008, 4096, "bf16", "w4a8")],
    "linear": [("bf16", 10240, 8192, 2048, "bf16", "normal", {"act": "gelu", "bias": True}),
               ("bf16", 597, 11008, 4096, "bf16", "normal", {"act": "silu", "gated": True}),
               ("fp8", 597, 11008, 4096, "bf16", "fp8", {"act": "silu", "gated": True})],
}


def workload_shapes(name: str):
    return list(WORKLOADS[name])


def make_workload_case(entry, seed: int = 0) -> GemmCase:
    dtype, m, n, k, out, dist = entry[:6]
    epi = entry[6] if len(entry) > 6 else {}
    rows_b = 2 * n if epi.get("gated") else n
    if dist == "square_normal":
        case = make_case(dtype, m, rows_b, k, out=out, dist="normal", seed=seed, a_std=1.0, b_std=1.0)
    else:
        case = make_case(dtype, m, rows_b, k, out=out, dist=dist, seed=seed)
    if epi:
        case.n = n
        case.gated = bool(epi.get("gated", False))
        case.act = ACT_IDS[epi.get("act", "none")]
        if epi.get("bias"):
            case.bias = normal(seed, STREAM_BIAS, (rows_b,), 0.0, 0.5).astype(np.float32)
        a_l, b_l = epi.get("layout", ("k", "k"))
        case.a_major, case.b_major = int(a_l == "mn"), int(b_l == "mn")
    return case
