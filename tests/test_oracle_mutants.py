"""Plant plausible mistakes in copies of the oracle (on the CPU) and check the pins catch each.

Each mutant is the oracle's C source with one textual edit, compiled into a
temporary library.  A mutant that every pin accepts would mean the pins cannot
tell that mistake from the real oracle.
"""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")

MUTANTS = {
    # a dropped term: the first k is skipped
    "drop_first_k": ("for (int64_t k = 0; k < K; ++k) {\n        double p = load_code",
                     "for (int64_t k = 1; k < K; ++k) {\n        double p = load_code"),
    # a dropped term: the last k is skipped
    "drop_last_k": ("for (int64_t k = 0; k < K; ++k) {\n        double p = load_code",
                    "for (int64_t k = 0; k + 1 < K; ++k) {\n        double p = load_code"),
    # a wrong sign in the accumulation
    "wrong_sign": ("load_code(dtype, B, j * K + k);\n        acc += p;", "load_code(dtype, B, j * K + k);\n        acc -= p;"),
    # a wrong index on B: k runs backwards along the row
    "reversed_k_on_B": ("load_code(dtype, B, j * K + k)", "load_code(dtype, B, j * K + (K - 1 - k))"),
    # a transposed operand read: B taken as [K, N] with the same buffer
    "b_as_column_major": ("load_code(dtype, B, j * K + k)", "load_code(dtype, B, (k * K + j) % (K * (j + 1)))"),
    # a dropped scale
    "drop_sb": ("double s = (double)sa[i] * (double)sb[j];", "double s = (double)sa[i];"),
    # scales applied by the wrong index
    "sa_by_col": ("double s = (double)sa[i] * (double)sb[j];", "double s = (double)sa[j % (i + 1)] * (double)sb[j];"),
    # decoder mistakes
    "bf16_bias": ("ldexp(1.0 + (double)frac / 128.0, expo - 127)", "ldexp(1.0 + (double)frac / 128.0, expo - 126)"),
    "e4m3_bias": ("ldexp(1.0 + (double)frac / 8.0, expo - 7)", "ldexp(1.0 + (double)frac / 8.0, expo - 8)"),
    "e4m3_subnormal": ("v = ldexp((double)frac / 8.0, 1 - 7);", "v = ldexp(1.0 + (double)frac / 8.0, -7);"),
    "e4m3_no_nan": ("if (expo == 0xF && frac == 0x7) {", "if (0) {"),
    # rounding mistakes
    "round_truncates": ("double r = nearbyint(a / q);", "double r = floor(a / q);"),
    "round_half_up": ("double r = nearbyint(a / q);", "double r = floor(a / q + 0.5);"),
    # magnitude sum wrong
    "mag_signed": ("acc += p;\n        mag += fabs(p);\n    }\n    if (sa && sb)", "acc += p;\n        mag += p;\n    }\n    if (sa && sb)"),
    # linear layer: activation constants and signs
    "gelu_half_not_root2": ("x * 0.5 * erfc(-x / sqrt(2.0))", "x * 0.5 * erfc(-x / 2.0)"),
    "gelu_sign": ("x * 0.5 * erfc(-x / sqrt(2.0))", "x * 0.5 * erfc(x / sqrt(2.0))"),
    "silu_sign": ("return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    # linear layer: bias and gate / up indexing
    "bias_dropped": ("const double x = g + bg;", "const double x = g;"),
    "bias_up_index": ("const double bu = bias ? (double)bias[n + j] : 0.0;", "const double bu = bias ? (double)bias[j] : 0.0;"),
    "up_row_is_gate_row": ("one_element(dtype, A, B, sa, sb, K, i, n + j, &u, &su);", "one_element(dtype, A, B, sa, sb, K, i, j, &u, &su);"),
    "gate_and_up_swapped": ("*y_out = ax * v;", "*y_out = oracle_act(act, v) * x;"),
    "error_scale_drops_bias": ("*e_out = L * (sg + fabs(bg));", "*e_out = L * sg;"),
    # block-scaled FP4: decoders, packing and block indexing
    "e2m1_bias": ("v = ldexp(1.0 + (double)frac / 2.0, expo - 1);", "v = ldexp(1.0 + (double)frac / 2.0, expo);"),
    "e2m1_subnormal_as_normal": ("v = ldexp((double)frac / 2.0, 1 - 1);", "v = ldexp(1.0 + (double)frac / 2.0, -1);"),
    "e2m1_sign_bit": ("int sign = (code >> 3) & 1;\n    int expo = (code >> 1) & 3;",
                      "int sign = (code >> 2) & 1;\n    int expo = (code >> 1) & 3;"),
    "e8m0_bias": ("return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 128);"),
    # (reading the high nibble first is an equivalent mutant: A and B swap the
    # same pair of elements of one block, so no product can tell; the packing
    # pins hold the byte index instead)
    "mx_bytes_reversed": ("uint8_t byte = X[r * (K / 2) + k / 2];", "uint8_t byte = X[r * (K / 2) + (K / 2 - 1 - k / 2)];"),
    "mx_drop_first_k": ("for (int64_t k = 0; k < K; ++k) {\n        double p = mx_value",
                        "for (int64_t k = 1; k < K; ++k) {\n        double p = mx_value"),
    "mx_drop_last_k": ("for (int64_t k = 0; k < K; ++k) {\n        double p = mx_value",
                       "for (int64_t k = 0; k + 1 < K; ++k) {\n        double p = mx_value"),
    "mx_blocks_of_64": ("E[r * (K / 32) + k / 32]", "E[r * (K / 32) + k / 64]"),
    "mx_scales_dropped": ("return oracle_decode_e8m0(E[r * (K / 32) + k / 32]) * oracle_decode_e2m1(code);",
                          "return oracle_decode_e2m1(code);"),
    "mx_mag_signed": ("double p = mx_value(A, EA, K, i, k) * mx_value(B, EB, K, j, k);\n        acc += p;\n        mag += fabs(p);",
                      "double p = mx_value(A, EA, K, i, k) * mx_value(B, EB, K, j, k);\n        acc += p;\n        mag += p;"),
    # W4A8: the weight nibble order (observable here: A is not packed), B's
    # row pitch, dropped terms and scales, the magnitude sum
    "w4_nibbles_swapped": ("return oracle_decode_e2m1((k % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4));",
                           "return oracle_decode_e2m1((k % 2 == 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4));"),
    "w4_row_pitch_K": ("uint8_t byte = B[j * (K / 2) + k / 2];", "uint8_t byte = B[j * K + k / 2];"),
    "w4_drop_first_k": ("for (int64_t k = 0; k < K; ++k) {\n        double p = oracle_decode_e4m3",
                        "for (int64_t k = 1; k < K; ++k) {\n        double p = oracle_decode_e4m3"),
    "w4_drop_last_k": ("for (int64_t k = 0; k < K; ++k) {\n        double p = oracle_decode_e4m3",
                       "for (int64_t k = 0; k + 1 < K; ++k) {\n        double p = oracle_decode_e4m3"),
    "w4_drop_sa": ("const double scale = (double)sa[i] * (double)sb[j];", "const double scale = (double)sb[j];"),
    "w4_a_index_transposed": ("oracle_decode_e4m3(A[i * K + k])", "oracle_decode_e4m3(A[(k * K + i) % (K * (i + 1))])"),
    "w4_mag_signed": ("*s_out = mag * fabs(scale);", "*s_out = acc * fabs(scale);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / f"{name}.c"
    mutant_src.write_text(src.replace(old, new))
    lib_path = str(tmp_path / f"lib{name}.so")
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", lib_path,
                    str(mutant_src), "-lm"], check=True)
    failed = oracle_pins.run_all(oracle.load(lib_path))
    assert failed, f"mutant {name} passes every pin"


def test_real_oracle_passes_every_pin():
    assert oracle_pins.run_all(oracle.load()) == []
