"""Checks that pin the oracle to facts other than itself.

Each check takes an oracle library handle, so the same checks run against the
oracle and against deliberately broken copies of it (tests/test_oracle_mutants.py).
A check raises AssertionError when the oracle disagrees with:
  - library decoders (torch bfloat16 / float8_e4m3fn -> float32) over every code,
  - values fixed by the formats (E4M3 max 448, smallest subnormal 2^-9, NaN code),
  - torch's float32 -> bfloat16 round-to-nearest-even,
  - closed forms: identity and permutation products, rank-1 outer products,
    all-ones, scaled rank-1,
  - brute force in exact rational arithmetic on tiny shapes,
  - for the linear layer: library routines for the normal distribution
    function and the logistic function, the symmetry act(x) - act(-x) = x,
    printed values (Phi(1), sigma(ln 3) = 3/4), and one-hot rows of A that
    turn the product into a lookup of B, so bias, gate and up terms are exact,
  - for the block-scaled FP4 (MXFP4) product: the E2M1 value table the format
    fixes, torch's E8M0 decoder over every code, hand-packed bytes whose
    product is known (which byte holds which element, which block scale
    covers which k), numpy's matmul when every scale is 1, and brute force in
    exact rational arithmetic.  (Which nibble of a byte comes first cannot
    change a product: A and B swap the same two elements of one block.)
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

import oracle
from synthetic import integers, to_bf16_codes, to_e4m3_codes


def _bf16(x):
    return to_bf16_codes(np.asarray(x, dtype=np.float64))


def check_bf16_decoder(lib):
    codes = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.decode_bf16(codes, lib=lib)
    want = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    with np.errstate(invalid="ignore"):  # signalling-NaN codes widen to quiet NaNs
        want = want.astype(np.float64)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), f"bf16 decoder differs at codes {codes[~same][:8]}"


def check_e4m3_decoder(lib):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(codes, lib=lib)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), f"e4m3 decoder differs at codes {codes[~same][:8]}"
    # values the format fixes
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9
    assert got[0x08] == 2.0 ** -6
    assert got[0x38] == 1.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert np.isfinite(np.delete(got, [0x7F, 0xFF])).all()


def check_round_bf16(lib):
    rng = np.random.default_rng(1234)
    # random float32 bit patterns over the finite range, plus exact ties
    bits = rng.integers(0, 0x7F7FFFFF, size=200000, dtype=np.uint32)
    x = bits.view(np.float32)
    x = np.concatenate([x, -x])
    ties = ((rng.integers(0x0080, 0x7F00, size=5000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, -0.0, 1.0, 3.0e38])])
    got = oracle.round_bf16(x.astype(np.float64), lib=lib)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = got != want
    assert not bad.any(), f"round_bf16 differs for {x[bad][:4]}: {got[bad][:4]} vs {want[bad][:4]}"


def check_identity(lib):
    K, n = 24, 40
    A = _bf16(np.eye(K))
    Bv = integers(7, 1, (n, K), -100, 100) / 8.0
    B = _bf16(Bv)
    C, S = oracle.gemm(oracle.BF16, A, B, lib=lib)
    assert C.shape == (K, n)
    np.testing.assert_array_equal(C, Bv.T)   # every k/8 with |k| <= 100 is exact in bf16
    np.testing.assert_array_equal(S, np.abs(Bv.T))


def check_permutation(lib):
    K, n, m = 16, 9, 12
    rng = np.random.default_rng(5)
    perm = rng.integers(0, K, size=m)
    P = np.zeros((m, K))
    P[np.arange(m), perm] = 1.0
    Bv = integers(3, 1, (n, K), -50, 50) / 4.0
    C, _ = oracle.gemm(oracle.BF16, _bf16(P), _bf16(Bv), lib=lib)
    np.testing.assert_array_equal(C, Bv[:, perm].T)


def check_rank1(lib):
    m, n, K = 7, 11, 33
    u = integers(11, 0, (m,), -3, 3)
    v = integers(11, 1, (n,), -3, 3)
    w = integers(11, 2, (K,), -4, 4)
    w2 = integers(11, 3, (K,), -4, 4)
    A = _bf16(np.outer(u, w))
    B = _bf16(np.outer(v, w2))
    C, _ = oracle.gemm(oracle.BF16, A, B, lib=lib)
    np.testing.assert_array_equal(C, np.outer(u, v) * float(np.dot(w, w2)))


def check_all_ones(lib):
    for dt, enc in ((oracle.BF16, _bf16), (oracle.E4M3, to_e4m3_codes)):
        m, n, K = 5, 6, 77
        C, S = oracle.gemm(dt, enc(np.ones((m, K))), enc(np.ones((n, K))),
                           *((np.ones(m, np.float32), np.ones(n, np.float32)) if dt == oracle.E4M3 else ()),
                           lib=lib)
        assert (C == K).all() and (S == K).all()


def check_scaled_rank1_e4m3(lib):
    m, n, K = 6, 10, 40
    u = integers(21, 0, (m,), -4, 4)
    v = integers(21, 1, (n,), -4, 4)
    w = integers(21, 2, (K,), -4, 4)
    w2 = integers(21, 3, (K,), -4, 4)
    sa = np.float32([0.5, 1, 2, 0.25, 4, 1.5])
    sb = np.linspace(0.5, 2.0, n).astype(np.float32)
    A = to_e4m3_codes(np.outer(u, w))
    B = to_e4m3_codes(np.outer(v, w2))
    C, S = oracle.gemm(oracle.E4M3, A, B, sa, sb, lib=lib)
    want = np.outer(u * sa.astype(np.float64), v * sb.astype(np.float64)) * float(np.dot(w, w2))
    np.testing.assert_array_equal(C, want)
    want_s = np.outer(np.abs(u) * sa, np.abs(v) * sb) * float(np.dot(np.abs(w), np.abs(w2)))
    np.testing.assert_allclose(S, want_s, rtol=1e-15)


def _exact_product(Av, Bv):
    m, K = Av.shape
    n = Bv.shape[0]
    out = np.empty((m, n), dtype=object)
    for i in range(m):
        for j in range(n):
            out[i, j] = sum((Fraction(float(Av[i, k])) * Fraction(float(Bv[j, k])) for k in range(K)),
                            Fraction(0))
    return out


def check_brute_force(lib):
    rng = np.random.default_rng(99)
    for trial in range(12):
        m, n, K = (int(x) for x in rng.integers(1, 9, size=3))
        A = _bf16(rng.normal(size=(m, K)))
        B = _bf16(rng.normal(size=(n, K)) * 3.0)
        Av = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).double().numpy()
        Bv = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).double().numpy()
        C, S = oracle.gemm(oracle.BF16, A, B, lib=lib)
        exact = _exact_product(Av, Bv)
        # bf16 x bf16 products are exact in double; K <= 8 sums of them stay exact
        for i in range(m):
            for j in range(n):
                assert Fraction(C[i, j]) == exact[i, j], (trial, i, j)
        np.testing.assert_array_equal(S, (np.abs(Av)[:, None, :] * np.abs(Bv)[None, :, :]).sum(-1))
    # e4m3 with scales
    for trial in range(6):
        m, n, K = (int(x) for x in rng.integers(1, 9, size=3))
        A = to_e4m3_codes(rng.normal(size=(m, K)) * 4)
        B = to_e4m3_codes(rng.normal(size=(n, K)))
        sa = rng.uniform(0.5, 2, size=m).astype(np.float32)
        sb = rng.uniform(0.5, 2, size=n).astype(np.float32)
        Av = torch.from_numpy(A).view(torch.float8_e4m3fn).double().numpy()
        Bv = torch.from_numpy(B).view(torch.float8_e4m3fn).double().numpy()
        C, _ = oracle.gemm(oracle.E4M3, A, B, sa, sb, lib=lib)
        exact = _exact_product(Av, Bv)
        for i in range(m):
            for j in range(n):
                want = exact[i, j] * Fraction(float(sa[i])) * Fraction(float(sb[j]))
                assert abs(Fraction(C[i, j]) - want) <= abs(want) * Fraction(1, 1 << 50), (trial, i, j)


def check_points_match_full(lib):
    m, n, K = 37, 29, 50
    A = _bf16(integers(4, 0, (m, K), -4, 4))
    B = _bf16(integers(4, 1, (n, K), -4, 4))
    C, S = oracle.gemm(oracle.BF16, A, B, lib=lib)
    rows = np.array([0, m - 1, 5, 36, 17])
    cols = np.array([0, n - 1, 28, 3, 11])
    Cp, Sp = oracle.gemm_points(oracle.BF16, A, B, rows, cols, lib=lib)
    np.testing.assert_array_equal(Cp, C[rows, cols])
    np.testing.assert_array_equal(Sp, S[rows, cols])


# ------------------------------------------------------------ the linear layer around the product
E4M3_ONE = 0x38  # 1.0 in E4M3: exponent field 7 (bias 7), fraction 0


def _ndtr(x):
    from scipy.special import ndtr  # standard normal distribution function, a library routine
    return ndtr(x)


def _expit(x):
    from scipy.special import expit  # the logistic function, a library routine
    return expit(x)


def _act_lib(kind, x):
    x = np.asarray(x, dtype=np.float64)
    if kind == oracle.ACT_GELU:
        return x * _ndtr(x)
    if kind == oracle.ACT_SILU:
        return x * _expit(x)
    return x


def check_act_closed_forms(lib):
    xs = np.array([-6.0, -3.0, -1.0, -0.5, -1e-3, 0.0, 1e-3, 0.5, 1.0, 2.0, 3.0, 6.0])
    for kind in (oracle.ACT_NONE, oracle.ACT_GELU, oracle.ACT_SILU):
        got = oracle.act(kind, xs, lib=lib)
        np.testing.assert_allclose(got, _act_lib(kind, xs), rtol=1e-13, atol=1e-300)
        if kind != oracle.ACT_NONE:
            # act(x) - act(-x) = x: Phi(x) + Phi(-x) = 1 and sigma(x) + sigma(-x) = 1
            np.testing.assert_allclose(got - oracle.act(kind, -xs, lib=lib), xs, rtol=1e-13, atol=1e-15)
    # printed table values: Phi(1) = 0.8413447..., sigma(ln 3) = 3/4 exactly
    assert abs(oracle.act(oracle.ACT_GELU, [1.0], lib=lib)[0] - 0.8413447460685429) < 1e-12
    ln3 = float(np.log(3.0))
    assert abs(oracle.act(oracle.ACT_SILU, [ln3], lib=lib)[0] - 0.75 * ln3) < 1e-15


def _one_hot_rows(m, K, seed):
    """A's rows are one-hot: row i has a single 1 at column k_i."""
    ks = integers(seed, 0, (m,), 0, K - 1).astype(np.int64)
    A = np.zeros((m, K))
    A[np.arange(m), ks] = 1.0
    return A, ks


def check_linear_bias_onehot(lib):
    m, n, K = 9, 13, 11
    A, ks = _one_hot_rows(m, K, 5)
    Bv = integers(5, 1, (n, K), -4, 4)
    bias = (integers(5, 2, (n,), -8, 8) / 4.0).astype(np.float32)  # exact quarters
    for kind in (oracle.ACT_NONE, oracle.ACT_GELU, oracle.ACT_SILU):
        Y, E = oracle.linear(oracle.BF16, _bf16(A), _bf16(Bv), bias=bias, act=kind, lib=lib)
        X = Bv[:, ks].T + bias[None, :].astype(np.float64)  # X[i, j] = B[j, k_i] + bias[j]
        np.testing.assert_allclose(Y, _act_lib(kind, X), rtol=1e-13, atol=1e-300)
        L = 1.0 if kind == oracle.ACT_NONE else 1.2
        np.testing.assert_allclose(E, L * (np.abs(Bv[:, ks].T) + np.abs(bias)[None, :]), rtol=1e-15)


def check_linear_gated_onehot(lib):
    m, n, K = 7, 10, 9
    A, ks = _one_hot_rows(m, K, 6)
    Bg = integers(6, 1, (n, K), -4, 4)
    Bu = integers(6, 3, (n, K), -4, 4)
    bias = (integers(6, 2, (2 * n,), -8, 8) / 4.0).astype(np.float32)
    for kind in (oracle.ACT_GELU, oracle.ACT_SILU):
        Y, E = oracle.linear(oracle.BF16, _bf16(A), _bf16(np.vstack([Bg, Bu])), bias=bias, act=kind,
                             gated=True, lib=lib)
        G = Bg[:, ks].T + bias[None, :n].astype(np.float64)
        U = Bu[:, ks].T + bias[None, n:].astype(np.float64)
        np.testing.assert_allclose(Y, _act_lib(kind, G) * U, rtol=1e-13, atol=1e-300)
        want_E = (np.abs(_act_lib(kind, G)) * (np.abs(Bu[:, ks].T) + np.abs(bias[None, n:]))
                  + 1.2 * np.abs(U) * (np.abs(Bg[:, ks].T) + np.abs(bias[None, :n])))
        np.testing.assert_allclose(E, want_E, rtol=1e-13, atol=1e-300)


def check_linear_gated_scaled_e4m3(lib):
    """E4M3 with per-row and per-column scales: the up half takes the scales and
    bias of rows n .. 2n-1 of B."""
    m, n, K = 6, 8, 16
    ks = integers(7, 0, (m,), 0, K - 1).astype(np.int64)
    A = np.zeros((m, K), dtype=np.uint8)
    A[np.arange(m), ks] = E4M3_ONE
    Bg = integers(7, 1, (n, K), -4, 4)
    Bu = integers(7, 3, (n, K), -4, 4)
    B = to_e4m3_codes(np.vstack([Bg, Bu]))
    pick = np.array([0.5, 1.0, 2.0], dtype=np.float32)
    sa = pick[integers(7, 4, (m,), 0, 2).astype(np.int64)]
    sb = pick[integers(7, 5, (2 * n,), 0, 2).astype(np.int64)]
    bias = (integers(7, 2, (2 * n,), -8, 8) / 4.0).astype(np.float32)
    Y, _ = oracle.linear(oracle.E4M3, A, B, sa, sb, bias=bias, act=oracle.ACT_SILU, gated=True, lib=lib)
    s_a = sa.astype(np.float64)[:, None]
    G = Bg[:, ks].T * s_a * sb[None, :n] + bias[None, :n]
    U = Bu[:, ks].T * s_a * sb[None, n:] + bias[None, n:]
    np.testing.assert_allclose(Y, _act_lib(oracle.ACT_SILU, G) * U, rtol=1e-13, atol=1e-300)


def check_linear_points_match_full(lib):
    m, n, K = 21, 17, 40
    A = _bf16(integers(8, 0, (m, K), -4, 4))
    B = _bf16(integers(8, 1, (2 * n, K), -4, 4))
    bias = (integers(8, 2, (2 * n,), -8, 8) / 8.0).astype(np.float32)
    Y, E = oracle.linear(oracle.BF16, A, B, bias=bias, act=oracle.ACT_GELU, gated=True, lib=lib)
    rows = np.array([0, m - 1, 4, 13])
    cols = np.array([0, n - 1, 16, 2])
    Yp, Ep = oracle.linear_points(oracle.BF16, A, B, rows, cols, bias=bias, act=oracle.ACT_GELU, gated=True, lib=lib)
    np.testing.assert_array_equal(Yp, Y[rows, cols])
    np.testing.assert_array_equal(Ep, E[rows, cols])


# ------------------------------------------------------------ block-scaled FP4 (MXFP4)
# E2M1 magnitudes of codes 0..7 as the format fixes them (OCP Microscaling
# version 1.0, table of FP4 E2M1 values); bit 3 is the sign
E2M1_TABLE = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}
E2M1_ONE = 0x2


def _e2m1_value(code):
    v = E2M1_TABLE[code & 7]
    return -v if code & 8 else v


def _unpack(packed):
    """[r, K/2] bytes -> [r, K] codes; element 2t is the low four bits of byte t."""
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def check_e2m1_decoder(lib):
    got = oracle.decode_e2m1(np.arange(16, dtype=np.uint8), lib=lib)
    for code in range(16):
        want = _e2m1_value(code)
        assert got[code] == want and np.signbit(got[code]) == (code >= 8), (code, got[code], want)


def check_e8m0_decoder(lib):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e8m0(codes, lib=lib)
    with np.errstate(invalid="ignore"):  # the NaN code widens to a quiet NaN
        want = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).float().numpy().astype(np.float64)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), f"e8m0 decoder differs at codes {codes[~same][:8]}"
    assert got[127] == 1.0 and got[128] == 2.0 and got[0] == 2.0 ** -127 and np.isnan(got[255])


def check_mx_nibble_order(lib):
    # B's row: element 0 is 0.5 (code 1), element 1 is 4.0 (code 6): byte 0 = 0x61
    K = 32
    B = np.zeros((1, K // 2), dtype=np.uint8)
    B[0, 0] = 0x61
    A = np.zeros((2, K // 2), dtype=np.uint8)
    A[0, 0] = E2M1_ONE          # element 0 is 1.0
    A[1, 0] = E2M1_ONE << 4     # element 1 is 1.0
    ones = np.full((2, 1), 127, dtype=np.uint8)
    C, S = oracle.mxfp4_gemm(A, B, ones, ones[:1], lib=lib)
    assert C[0, 0] == 0.5 and C[1, 0] == 4.0, C
    assert S[0, 0] == 0.5 and S[1, 0] == 4.0


def check_mx_block_scales(lib):
    # all elements 1.0 over K = 96 (three blocks); C = 32 * sum_b 2^(ea_b - 127) 2^(eb_b - 127)
    K = 96
    ones_byte = E2M1_ONE | (E2M1_ONE << 4)
    A = np.full((2, K // 2), ones_byte, dtype=np.uint8)
    B = np.full((2, K // 2), ones_byte, dtype=np.uint8)
    EA = np.array([[127, 130, 127], [126, 127, 129]], dtype=np.uint8)
    EB = np.array([[127, 127, 127], [129, 125, 127]], dtype=np.uint8)
    C, _ = oracle.mxfp4_gemm(A, B, EA, EB, lib=lib)
    for i in range(2):
        for j in range(2):
            want = 32 * sum(2.0 ** (int(EA[i, b]) - 127) * 2.0 ** (int(EB[j, b]) - 127) for b in range(3))
            assert C[i, j] == want, (i, j, C[i, j], want)
    # one element at k = 33 (block 1, the high nibble of byte 16) picks block 1's scales only
    A1 = np.zeros((1, K // 2), dtype=np.uint8)
    A1[0, 16] = E2M1_ONE << 4
    C1, _ = oracle.mxfp4_gemm(A1, B[:1], EA[:1], EB[1:], lib=lib)
    assert C1[0, 0] == 2.0 ** 3 * 2.0 ** -2


def check_mx_unit_scales_match_matmul(lib):
    rng = np.random.default_rng(7)
    m, n, K = 9, 11, 160
    A = rng.integers(0, 256, size=(m, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
    C, S = oracle.mxfp4_gemm(A, B, np.full((m, K // 32), 127, np.uint8), np.full((n, K // 32), 127, np.uint8),
                             lib=lib)
    Av = np.vectorize(_e2m1_value)(_unpack(A))
    Bv = np.vectorize(_e2m1_value)(_unpack(B))
    np.testing.assert_array_equal(C, Av @ Bv.T)   # multiples of 1/4 below 2^12: exact in double
    np.testing.assert_array_equal(S, np.abs(Av) @ np.abs(Bv).T)


def check_mx_brute_force(lib):
    rng = np.random.default_rng(31)
    for trial in range(10):
        m, n = (int(x) for x in rng.integers(1, 6, size=2))
        K = 32 * int(rng.integers(1, 4))
        A = rng.integers(0, 256, size=(m, K // 2), dtype=np.uint8)
        B = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
        EA = rng.integers(115, 140, size=(m, K // 32), dtype=np.uint8)
        EB = rng.integers(115, 140, size=(n, K // 32), dtype=np.uint8)
        C, _ = oracle.mxfp4_gemm(A, B, EA, EB, lib=lib)
        Ac, Bc = _unpack(A), _unpack(B)
        for i in range(m):
            for j in range(n):
                want = sum((Fraction(_e2m1_value(int(Ac[i, k]))) * Fraction(2) ** (int(EA[i, k // 32]) - 127) *
                            Fraction(_e2m1_value(int(Bc[j, k]))) * Fraction(2) ** (int(EB[j, k // 32]) - 127)
                            for k in range(K)), Fraction(0))
                assert Fraction(C[i, j]) == want, (trial, i, j)


def check_mx_points_match_full(lib):
    rng = np.random.default_rng(5)
    m, n, K = 13, 17, 64
    A = rng.integers(0, 256, size=(m, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
    EA = rng.integers(120, 135, size=(m, K // 32), dtype=np.uint8)
    EB = rng.integers(120, 135, size=(n, K // 32), dtype=np.uint8)
    C, S = oracle.mxfp4_gemm(A, B, EA, EB, lib=lib)
    rows = np.array([0, m - 1, 4, 12])
    cols = np.array([0, n - 1, 16, 9])
    Cp, Sp = oracle.mxfp4_gemm_points(A, B, EA, EB, rows, cols, lib=lib)
    np.testing.assert_array_equal(Cp, C[rows, cols])
    np.testing.assert_array_equal(Sp, S[rows, cols])


# ------------------------------------------------------------ W4A8: E4M3 activations x E2M1 weights
def _e4m3_values(codes):
    """E4M3 codes -> float64 through torch's float8_e4m3fn (a library decoder)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def check_w4a8_nibble_order_and_scales(lib):
    # A one-hot: row i holds 1.0 at k = i, so C[i, j] = sa[i] sb[j] e2m1(B[j, i]);
    # element 2t of a B row is the low four bits of byte t
    K = 32
    A = np.zeros((4, K), dtype=np.uint8)
    for i in range(4):
        A[i, i] = E4M3_ONE
    B = np.zeros((2, K // 2), dtype=np.uint8)
    B[0, 0] = 0x61            # k = 0: 0.5 (code 1), k = 1: 4.0 (code 6)
    B[0, 1] = 0xA7            # k = 2: 6.0 (code 7), k = 3: -1.0 (code 0xA)
    B[1, 0] = 0x5D            # k = 0: -3.0 (code 0xD), k = 1: 3.0 (code 5)
    B[1, 1] = 0x0F            # k = 2: -6.0 (code 0xF), k = 3: 0
    sa = np.array([1.0, 2.0, 0.5, 4.0], dtype=np.float32)
    sb = np.array([1.0, 0.25], dtype=np.float32)
    C, S = oracle.w4a8_gemm(A, B, sa, sb, lib=lib)
    vals = [[0.5, 4.0, 6.0, -1.0], [-3.0, 3.0, -6.0, 0.0]]
    for i in range(4):
        for j in range(2):
            assert C[i, j] == sa[i] * sb[j] * vals[j][i], (i, j, C[i, j])
            assert S[i, j] == abs(sa[i] * sb[j] * vals[j][i])


def check_w4a8_brute_force(lib):
    rng = np.random.default_rng(41)
    for trial in range(10):
        m, n = (int(x) for x in rng.integers(1, 6, size=2))
        K = 2 * int(rng.integers(1, 40))
        A = rng.integers(0, 256, size=(m, K), dtype=np.uint8)
        A[(A & 0x7F) == 0x7F] = 0x3C          # no NaN codes
        B = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
        sa = (2.0 ** rng.integers(-3, 4, size=m)).astype(np.float32)
        sb = (2.0 ** rng.integers(-3, 4, size=n)).astype(np.float32)
        C, _ = oracle.w4a8_gemm(A, B, sa, sb, lib=lib)
        Av = _e4m3_values(A)
        Bc = _unpack(B)
        for i in range(m):
            for j in range(n):
                want = sum((Fraction(float(Av[i, k])) * Fraction(_e2m1_value(int(Bc[j, k]))) for k in range(K)),
                           Fraction(0)) * Fraction(float(sa[i])) * Fraction(float(sb[j]))
                assert Fraction(C[i, j]) == want, (trial, i, j)


def check_w4a8_matches_e4m3_product(lib):
    # every E2M1 value is an E4M3 value: re-encoding B as E4M3 codes gives the
    # same products in the same order, so the E4M3 product (pinned above)
    # must agree bit for bit
    rng = np.random.default_rng(43)
    m, n, K = 7, 9, 96
    A = rng.integers(0, 256, size=(m, K), dtype=np.uint8)
    A[(A & 0x7F) == 0x7F] = 0xB8
    B = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
    sa = rng.uniform(0.5, 2.0, size=m).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, size=n).astype(np.float32)
    Bv = np.vectorize(_e2m1_value)(_unpack(B))
    B8 = torch.from_numpy(Bv.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (_e4m3_values(B8) == Bv).all()
    C, S = oracle.w4a8_gemm(A, B, sa, sb, lib=lib)
    C8, S8 = oracle.gemm(oracle.E4M3, A, B8, sa, sb, lib=lib)
    np.testing.assert_array_equal(C, C8)
    np.testing.assert_array_equal(S, S8)


def check_w4a8_points_match_full(lib):
    rng = np.random.default_rng(47)
    m, n, K = 11, 13, 64
    A = rng.integers(0, 0x70, size=(m, K), dtype=np.uint8)
    B = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
    sa = rng.uniform(0.5, 2.0, size=m).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, size=n).astype(np.float32)
    C, S = oracle.w4a8_gemm(A, B, sa, sb, lib=lib)
    rows = np.array([0, m - 1, 3, 10])
    cols = np.array([0, n - 1, 12, 5])
    Cp, Sp = oracle.w4a8_gemm_points(A, B, sa, sb, rows, cols, lib=lib)
    np.testing.assert_array_equal(Cp, C[rows, cols])
    np.testing.assert_array_equal(Sp, S[rows, cols])


ALL_CHECKS = [check_bf16_decoder, check_e4m3_decoder, check_round_bf16, check_identity,
              check_permutation, check_rank1, check_all_ones, check_scaled_rank1_e4m3,
              check_brute_force, check_points_match_full, check_act_closed_forms, check_linear_bias_onehot,
              check_linear_gated_onehot, check_linear_gated_scaled_e4m3, check_linear_points_match_full,
              check_e2m1_decoder, check_e8m0_decoder, check_mx_nibble_order, check_mx_block_scales,
              check_mx_unit_scales_match_matmul, check_mx_brute_force, check_mx_points_match_full,
              check_w4a8_nibble_order_and_scales, check_w4a8_brute_force, check_w4a8_matches_e4m3_product,
              check_w4a8_points_match_full]


def run_all(lib):
    """Run every check; return the names of those that failed."""
    failed = []
    for chk in ALL_CHECKS:
        try:
            chk(lib)
        except AssertionError:
            failed.append(chk.__name__)
    return failed
