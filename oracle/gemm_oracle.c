/*
 * Reference oracle for the dense linear-layer GEMM  C[i,j] = sum_k A[i,k] * B[j,k].
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA path.
 *
 * What it computes (plain definition, no blocking, no reordering):
 *   - The product of a linear layer flattened to one GEMM: rows i of A are the
 *     tokens (M = B*L), rows j of B are the weight rows W[d_ff, d_model], and
 *     K = d_model is the shared inner dimension
 *     ("GEMM analysis in TraceLens", sections "Linear layers in LLMs" and
 *      "Flattening for GEMM": Y = X_flat @ W^T).
 *   - The operand orientation A[M,K] x B[N,K]^T with B stored [N,K]
 *     ("Gemm Optimization" guide, section 1.1 "Three-Level Tiling").
 *   - For 8-bit inputs the accumulator is multiplied by a per-row scale of A
 *     and a per-column scale of B ("Gemm Optimization" guide, section 7.1
 *     "Direct Store": value = acc * scale_a * scale_b).
 *
 * Arithmetic: every input code is decoded exactly into a double, products and
 * sums are formed in double in ascending k, one (i, j) at a time.  The sum of
 * absolute products S[i,j] = sum_k |a_ik * b_jk| (times |sa_i * sb_j|) is
 * returned beside the value for the tolerance test.
 *
 * Decoders are written from the format definitions:
 *   bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 *   E4M3 (OCP "E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 *   bits, no infinities, S.1111.111 is NaN, largest finite 448.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_E4M3 1

double oracle_decode_bf16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xFF;
    int frac = bits & 0x7F;
    double v;
    if (expo == 0xFF) {
        v = frac ? NAN : INFINITY;
    } else if (expo == 0) {
        /* subnormal: 0.fraction * 2^(1-127) */
        v = ldexp((double)frac / 128.0, 1 - 127);
    } else {
        v = ldexp(1.0 + (double)frac / 128.0, expo - 127);
    }
    return sign ? -v : v;
}

double oracle_decode_e4m3(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int frac = code & 0x7;
    double v;
    if (expo == 0xF && frac == 0x7) {
        v = NAN;
    } else if (expo == 0) {
        /* subnormal: 0.fraction * 2^(1-7) */
        v = ldexp((double)frac / 8.0, 1 - 7);
    } else {
        v = ldexp(1.0 + (double)frac / 8.0, expo - 7);
    }
    return sign ? -v : v;
}

/*
 * Round a double to the nearest bfloat16, ties to even, and return its bit
 * pattern.  This is the rounding the output cast is read to use (the pages do
 * not name one; round-to-nearest-even is the IEEE default).
 */
uint16_t oracle_round_bf16(double x)
{
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000 : 0);
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int unbiased = e - 1;         /* a = g * 2^unbiased, g in [1, 2) */
    if (unbiased < -126) unbiased = -126;   /* subnormal range: fixed quantum */
    /* quantum of the 7-bit fraction at this binade */
    double q = ldexp(1.0, unbiased - 7);
    double r = nearbyint(a / q);  /* current rounding mode: nearest, ties to even */
    double v = r * q;
    if (v == 0.0) return sign;    /* rounded below half the smallest subnormal */
    /* rounding may carry into the next binade; re-derive the fields from v */
    if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    int ev;
    frexp(v, &ev);
    int ub = ev - 1;
    uint16_t bits;
    if (ub < -126) {
        /* subnormal: v = frac * 2^-133 */
        bits = (uint16_t)(int)nearbyint(v / ldexp(1.0, -133));
    } else {
        int frac = (int)nearbyint((v / ldexp(1.0, ub) - 1.0) * 128.0);
        bits = (uint16_t)(((ub + 127) << 7) | frac);
    }
    return (uint16_t)(sign | bits);
}

/* Element-wise oracle_round_bf16 over an array. */
void oracle_round_bf16_n(const double* x, int64_t count, uint16_t* out)
{
    for (int64_t t = 0; t < count; ++t) out[t] = oracle_round_bf16(x[t]);
}

static double load_code(int dtype, const void* base, int64_t idx)
{
    if (dtype == ORACLE_BF16)
        return oracle_decode_bf16(((const uint16_t*)base)[idx]);
    return oracle_decode_e4m3(((const uint8_t*)base)[idx]);
}

/* One output element, by the definition. */
static void one_element(int dtype, const void* A, const void* B,
                        const float* sa, const float* sb, int64_t K,
                        int64_t i, int64_t j, double* c_out, double* s_out)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = load_code(dtype, A, i * K + k) * load_code(dtype, B, j * K + k);
        acc += p;
        mag += fabs(p);
    }
    if (sa && sb) {
        double s = (double)sa[i] * (double)sb[j];
        acc *= s;
        mag *= fabs(s);
    }
    *c_out = acc;
    *s_out = mag;
}

/*
 * Full product over the valid region.
 *   A: m rows of K codes (row-major), B: n rows of K codes (row-major).
 *   sa[m], sb[n]: fp32 scales, or both NULL for the unscaled product.
 *   C_ref[m*n], S_abs[m*n]: row-major outputs (S_abs may be NULL).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm(int dtype, const void* A, const void* B,
                const float* sa, const float* sb,
                int64_t m, int64_t n, int64_t K,
                double* C_ref, double* S_abs)
{
    if ((dtype != ORACLE_BF16 && dtype != ORACLE_E4M3) || !A || !B || !C_ref ||
        m < 0 || n < 0 || K < 0 || ((sa == NULL) != (sb == NULL)))
        return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double c, s;
            one_element(dtype, A, B, sa, sb, K, i, j, &c, &s);
            C_ref[i * n + j] = c;
            if (S_abs) S_abs[i * n + j] = s;
        }
    }
    return 0;
}

/*
 * The same definition at a list of (row, col) points, for products too large
 * to form in full.  rows[p] < m and cols[p] < n are the caller's contract;
 * out-of-range points return -1 before any work.
 */
int oracle_gemm_points(int dtype, const void* A, const void* B,
                       const float* sa, const float* sb,
                       int64_t m, int64_t n, int64_t K,
                       const int64_t* rows, const int64_t* cols, int64_t npts,
                       double* C_ref, double* S_abs)
{
    if ((dtype != ORACLE_BF16 && dtype != ORACLE_E4M3) || !A || !B || !C_ref ||
        !rows || !cols || npts < 0 || ((sa == NULL) != (sb == NULL)))
        return -1;
    for (int64_t p = 0; p < npts; ++p)
        if (rows[p] < 0 || rows[p] >= m || cols[p] < 0 || cols[p] >= n) return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t p = 0; p < npts; ++p) {
        double c, s;
        one_element(dtype, A, B, sa, sb, K, rows[p], cols[p], &c, &s);
        C_ref[p] = c;
        if (S_abs) S_abs[p] = s;
    }
    return 0;
}

/*
 * ---- The linear layer around the product ------------------------------------
 *
 * A linear layer adds a bias per output feature to the product, Y = X W^T + b
 * ("GEMM analysis in TraceLens", section "Backward pass GEMMs": the forward
 * operation Y = X @ W^T + b, whose bias gradient db has shape [d_ff]; the
 * trace's aten::addmm is that call).  A feed-forward block applies an
 * activation to the first projection (Funlib GEMM issue, section
 * "Description": XW1 -> GELU -> XW2), and the LLaMA MLP pairs an up and a gate
 * projection of the same shape ("GEMM analysis in TraceLens", section
 * "Real-world example: LLaMA-2 7B").
 *
 *   act 0: identity;  act 1: GELU(x) = x * Phi(x), Phi the standard normal
 *   distribution function (the exact, erf form);  act 2: SiLU(x) = x * sigma(x),
 *   sigma the logistic function.
 *
 *   plain:  Y[i,j] = act(c(i, j) + bias[j])
 *   gated:  Y[i,j] = act(c(i, j) + bias[j]) * (c(i, n + j) + bias[n + j])
 *           B holds 2n rows: the gate projection's n rows, then the up
 *           projection's n rows; sb and bias hold 2n entries in the same order.
 * where c(i, r) is the (scaled) product of row i of A with row r of B as
 * above, and bias may be NULL (all zeros).
 *
 * E_abs is the error scale of the tolerance test: how far Y may move when
 * each product moves by its own allowance (which scales with S + |bias|).
 * Plain: L * (S + |b|), with L = 1.2 bounding |act'| (GELU' <= 1.13,
 * SiLU' <= 1.10).  Gated: |act(g)| * (S_up + |b_up|) + L * |u| * (S_g + |b_g|),
 * to first order in the allowances.
 */
#define ORACLE_ACT_NONE 0
#define ORACLE_ACT_GELU 1
#define ORACLE_ACT_SILU 2

double oracle_act(int act, double x)
{
    switch (act) {
    case ORACLE_ACT_GELU: return x * 0.5 * erfc(-x / sqrt(2.0));   /* Phi(x) = erfc(-x / sqrt 2) / 2 */
    case ORACLE_ACT_SILU: return x / (1.0 + exp(-x));
    default: return x;
    }
}

static double act_slope_bound(int act)
{
    return act == ORACLE_ACT_NONE ? 1.0 : 1.2;
}

static void linear_element(int dtype, const void* A, const void* B,
                           const float* sa, const float* sb, const float* bias,
                           int64_t n, int64_t K, int act, int gated,
                           int64_t i, int64_t j, double* y_out, double* e_out)
{
    double g, sg;
    one_element(dtype, A, B, sa, sb, K, i, j, &g, &sg);
    const double bg = bias ? (double)bias[j] : 0.0;
    const double x = g + bg;
    const double ax = oracle_act(act, x);
    const double L = act_slope_bound(act);
    if (!gated) {
        *y_out = ax;
        *e_out = L * (sg + fabs(bg));
        return;
    }
    double u, su;
    one_element(dtype, A, B, sa, sb, K, i, n + j, &u, &su);
    const double bu = bias ? (double)bias[n + j] : 0.0;
    const double v = u + bu;
    *y_out = ax * v;
    *e_out = fabs(ax) * (su + fabs(bu)) + L * fabs(v) * (sg + fabs(bg));
}

static int linear_args_ok(int dtype, const void* A, const void* B, const float* sa, const float* sb,
                          int64_t m, int64_t n, int64_t K, int act, int gated, const double* Y)
{
    return (dtype == ORACLE_BF16 || dtype == ORACLE_E4M3) && A && B && Y && m >= 0 && n >= 0 &&
           K >= 0 && (sa == NULL) == (sb == NULL) && act >= ORACLE_ACT_NONE && act <= ORACLE_ACT_SILU &&
           (gated == 0 || gated == 1);
}

/*
 * The linear layer over the valid region: Y_ref[m*n] and E_abs[m*n]
 * (row-major; E_abs may be NULL).  B has n rows (2n when gated).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_linear(int dtype, const void* A, const void* B,
                  const float* sa, const float* sb, const float* bias,
                  int64_t m, int64_t n, int64_t K, int act, int gated,
                  double* Y_ref, double* E_abs)
{
    if (!linear_args_ok(dtype, A, B, sa, sb, m, n, K, act, gated, Y_ref)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double y, e;
            linear_element(dtype, A, B, sa, sb, bias, n, K, act, gated, i, j, &y, &e);
            Y_ref[i * n + j] = y;
            if (E_abs) E_abs[i * n + j] = e;
        }
    }
    return 0;
}

/* The linear layer at a list of (row, col) points; as oracle_gemm_points. */
int oracle_linear_points(int dtype, const void* A, const void* B,
                         const float* sa, const float* sb, const float* bias,
                         int64_t m, int64_t n, int64_t K, int act, int gated,
                         const int64_t* rows, const int64_t* cols, int64_t npts,
                         double* Y_ref, double* E_abs)
{
    if (!linear_args_ok(dtype, A, B, sa, sb, m, n, K, act, gated, Y_ref) || !rows || !cols || npts < 0)
        return -1;
    for (int64_t p = 0; p < npts; ++p)
        if (rows[p] < 0 || rows[p] >= m || cols[p] < 0 || cols[p] >= n) return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t p = 0; p < npts; ++p) {
        double y, e;
        linear_element(dtype, A, B, sa, sb, bias, n, K, act, gated, rows[p], cols[p], &y, &e);
        Y_ref[p] = y;
        if (E_abs) E_abs[p] = e;
    }
    return 0;
}

/*
 * ---- Block-scaled FP4 (MXFP4) ------------------------------------------------
 *
 * The "Gemm Optimization" guide's bandwidth formulas (section 8.2, "FP4
 * (MXFP4)") count half a byte per element of A and of B plus one byte per 32
 * elements of K for every row of A and every row of B.  The page names the
 * format and nothing more; the reading taken is the OCP Microscaling format
 * it names: E2M1 elements, and one E8M0 scale for each block of 32
 * consecutive elements of a row along K, so that
 *   value(X, r, k) = 2^(E[r, k / 32] - 127) * e2m1(X[r, k])
 *   C[i,j] = sum_k value(A, i, k) * value(B, j, k)
 * Storage: X holds K / 2 bytes per row, element 2t in the low four bits of
 * byte t and element 2t + 1 in the high four; E holds K / 32 bytes per row.
 * K must be a multiple of 32 (whole blocks).
 *
 * Decoders from the format definitions:
 *   E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 fraction bit; exponent 0 is
 *   subnormal (fraction * 2^-1); no infinities or NaN; largest magnitude 6.
 *   E8M0: 8 exponent bits (bias 127), no sign or fraction; 0xFF is NaN.
 */
double oracle_decode_e2m1(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int expo = (code >> 1) & 3;
    int frac = code & 1;
    double v;
    if (expo == 0)
        v = ldexp((double)frac / 2.0, 1 - 1);          /* subnormal: 0.f * 2^(1-1) */
    else
        v = ldexp(1.0 + (double)frac / 2.0, expo - 1);
    return sign ? -v : v;
}

double oracle_decode_e8m0(uint8_t code)
{
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

static double mx_value(const uint8_t* X, const uint8_t* E, int64_t K, int64_t r, int64_t k)
{
    uint8_t byte = X[r * (K / 2) + k / 2];
    uint8_t code = (k % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
    return oracle_decode_e8m0(E[r * (K / 32) + k / 32]) * oracle_decode_e2m1(code);
}

static void mx_element(const uint8_t* A, const uint8_t* B, const uint8_t* EA, const uint8_t* EB,
                       int64_t K, int64_t i, int64_t j, double* c_out, double* s_out)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = mx_value(A, EA, K, i, k) * mx_value(B, EB, K, j, k);
        acc += p;
        mag += fabs(p);
    }
    *c_out = acc;
    *s_out = mag;
}

/*
 * Full MXFP4 product over the valid region: A [m][K/2], B [n][K/2] packed
 * E2M1 codes, EA [m][K/32], EB [n][K/32] E8M0 scales; C_ref and S_abs
 * [m*n] row-major (S_abs may be NULL).  Returns 0, or -1 on a bad argument.
 */
int oracle_mxfp4_gemm(const uint8_t* A, const uint8_t* B, const uint8_t* EA, const uint8_t* EB,
                      int64_t m, int64_t n, int64_t K, double* C_ref, double* S_abs)
{
    if (!A || !B || !EA || !EB || !C_ref || m < 0 || n < 0 || K < 0 || K % 32 != 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double c, s;
            mx_element(A, B, EA, EB, K, i, j, &c, &s);
            C_ref[i * n + j] = c;
            if (S_abs) S_abs[i * n + j] = s;
        }
    }
    return 0;
}

/* The MXFP4 product at a list of (row, col) points; as oracle_gemm_points. */
int oracle_mxfp4_gemm_points(const uint8_t* A, const uint8_t* B, const uint8_t* EA, const uint8_t* EB,
                             int64_t m, int64_t n, int64_t K, const int64_t* rows, const int64_t* cols,
                             int64_t npts, double* C_ref, double* S_abs)
{
    if (!A || !B || !EA || !EB || !C_ref || !rows || !cols || npts < 0 || m < 0 || n < 0 || K < 0 ||
        K % 32 != 0)
        return -1;
    for (int64_t p = 0; p < npts; ++p)
        if (rows[p] < 0 || rows[p] >= m || cols[p] < 0 || cols[p] >= n) return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t p = 0; p < npts; ++p) {
        double c, s;
        mx_element(A, B, EA, EB, K, rows[p], cols[p], &c, &s);
        C_ref[p] = c;
        if (S_abs) S_abs[p] = s;
    }
    return 0;
}

/*
 * ---- 8-bit activations, 4-bit weights (W4A8) ----------------------------------
 *
 * The "Gemm Optimization" guide's bandwidth formulas (section 8.2) give, for
 * its "INT4" case, one byte per element of A, half a byte per element of B,
 * a bf16 C and (M + N) fp32 scales: 8-bit activations with a per-token scale
 * and 4-bit weights with a per-output-channel scale.  Reading taken: A holds
 * E4M3 codes (the 8-bit type the FP8/INT8 formula above it counts) with a
 * per-row scale sa; B holds 4-bit E2M1 codes, two per byte (element 2t in the
 * low four bits of byte t), with a per-row scale sb (one per column of C):
 *   C[i,j] = sa[i] * sb[j] * sum_k e4m3(A[i,k]) * e2m1(B[j,k])
 * in the order of the E4M3 product above (the sum first, then sa * sb).
 * A: m rows of K bytes; B: n rows of K / 2 bytes; K even.
 */
static double w4_value(const uint8_t* B, int64_t K, int64_t j, int64_t k)
{
    uint8_t byte = B[j * (K / 2) + k / 2];
    return oracle_decode_e2m1((k % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4));
}

static void w4a8_element(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb, int64_t K,
                         int64_t i, int64_t j, double* c_out, double* s_out)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = oracle_decode_e4m3(A[i * K + k]) * w4_value(B, K, j, k);
        acc += p;
        mag += fabs(p);
    }
    const double scale = (double)sa[i] * (double)sb[j];
    *c_out = acc * scale;
    *s_out = mag * fabs(scale);
}

/*
 * Full W4A8 product over the valid region: A [m][K] E4M3 codes, B [n][K/2]
 * packed E2M1 codes, sa [m], sb [n] fp32 scales; C_ref and S_abs [m*n]
 * row-major (S_abs may be NULL).  Returns 0, or -1 on a bad argument.
 */
int oracle_w4a8_gemm(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                     int64_t m, int64_t n, int64_t K, double* C_ref, double* S_abs)
{
    if (!A || !B || !sa || !sb || !C_ref || m < 0 || n < 0 || K < 0 || K % 2 != 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double c, s;
            w4a8_element(A, B, sa, sb, K, i, j, &c, &s);
            C_ref[i * n + j] = c;
            if (S_abs) S_abs[i * n + j] = s;
        }
    }
    return 0;
}

/* The W4A8 product at a list of (row, col) points; as oracle_gemm_points. */
int oracle_w4a8_gemm_points(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                            int64_t m, int64_t n, int64_t K, const int64_t* rows, const int64_t* cols,
                            int64_t npts, double* C_ref, double* S_abs)
{
    if (!A || !B || !sa || !sb || !C_ref || !rows || !cols || npts < 0 || m < 0 || n < 0 || K < 0 || K % 2 != 0)
        return -1;
    for (int64_t p = 0; p < npts; ++p)
        if (rows[p] < 0 || rows[p] >= m || cols[p] < 0 || cols[p] >= n) return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t p = 0; p < npts; ++p) {
        double c, s;
        w4a8_element(A, B, sa, sb, K, rows[p], cols[p], &c, &s);
        C_ref[p] = c;
        if (S_abs) S_abs[p] = s;
    }
    return 0;
}

/* Threads an OpenMP region of this library uses (1 without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
