/*
 * swiglu_oracle.c -- plain, slow, double-precision CPU oracle for the fused
 * SwiGLU projection.  TEST INFRASTRUCTURE ONLY: only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load this code.  It shares no
 * code, header or constant with the CUDA path.
 *
 * What it computes (page "Riepilogo Tecnico: Sovrapposizione delle Attivazioni
 * a Livello di Tile per l'Inferenza Efficiente di LLM", gist.science paper
 * 2607.02521, section "Definizione del Problema"):
 *
 *     Y = SiLU(A x W1) (.) (A x W2)
 *
 * with A[M,K], W1[K,N], W2[K,N]; two independent matrix products followed by
 * an element-wise gate.  The interleaved form (same page, section
 * "Metodologia", item 2 "Kernel-2: Interleave SwiGLU") stores W1 and W2 as
 * one W_fused[K,2N] whose even column 2n is gate column n and whose odd column
 * 2n+1 is up column n; a single product D = A x W_fused is followed by
 * Y[m,n] = SiLU(D[m,2n]) * D[m,2n+1].
 *
 * Readings taken where the page is silent (each is listed in the design notes):
 *   - SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x)) (Swish with beta = 1);
 *   - the weights are row-major [K,N] (the page writes A x W1 and K x 2N);
 *   - the products are accumulated exactly as written, k = 0..K-1, in double,
 *     over the exact values of the BF16 (or dequantised FP8) inputs;
 *   - G and U are never rounded; Y is returned unrounded in double.
 *
 * Every function processes the rows listed in `rows` (or all M rows when
 * rows == NULL), so that very large shapes can be checked on a row sample.
 * Rows are independent (row m of Y depends only on row m of A), so splitting
 * them over OpenMP threads does not change any result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- element decoding ------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32: widen the 16 bits to 32 and
 * read the result as a float (exact), then as a double (exact). */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* FP8 E4M3 ("fn" variant, OCP 8-bit floating point): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
 * (value = mantissa/8 * 2^-6); S.1111.111 is NaN; there are no infinities,
 * so the largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_f64(uint8_t bits)
{
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* SiLU(x) = x * sigmoid(x) = x / (1 + e^-x). */
double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* ---- the definition, separate weights --------------------------------- */

/* Row r of the products: g[n] = sum_k a[k] W1[k,n], u[n] = sum_k a[k] W2[k,n].
 * a, w1, w2 are already decoded to double. */
static void gate_up_row(const double *a, const double *w1, const double *w2,
                        int64_t N, int64_t K, double *g, double *u)
{
    for (int64_t n = 0; n < N; ++n) {
        g[n] = 0.0;
        u[n] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
        const double ak = a[k];
        const double *w1k = w1 + k * N;
        const double *w2k = w2 + k * N;
        for (int64_t n = 0; n < N; ++n) {
            g[n] += ak * w1k[n];
            u[n] += ak * w2k[n];
        }
    }
}

static double *decode_bf16_matrix(const uint16_t *x, int64_t count)
{
    double *d = (double *)malloc((size_t)(count > 0 ? count : 1) * sizeof(double));
    if (!d)
        return NULL;
    for (int64_t i = 0; i < count; ++i)
        d[i] = oracle_bf16_to_f64(x[i]);
    return d;
}

static double *decode_e4m3_matrix(const uint8_t *x, int64_t count, double scale)
{
    double *d = (double *)malloc((size_t)(count > 0 ? count : 1) * sizeof(double));
    if (!d)
        return NULL;
    for (int64_t i = 0; i < count; ++i)
        d[i] = oracle_e4m3_to_f64(x[i]) * scale;
    return d;
}

/* Row m of A, decoded to double: kind 0 = BF16 bit patterns, kind 1 = E4M3
 * codes times the per-tensor scale sA. */
static void decode_a_row(const void *A, int kind, double sA, int64_t m,
                         int64_t K, double *a)
{
    if (kind == 0) {
        const uint16_t *r = (const uint16_t *)A + m * K;
        for (int64_t k = 0; k < K; ++k)
            a[k] = oracle_bf16_to_f64(r[k]);
    } else {
        const uint8_t *r = (const uint8_t *)A + m * K;
        for (int64_t k = 0; k < K; ++k)
            a[k] = oracle_e4m3_to_f64(r[k]) * sA;
    }
}

/* Shared driver: A raw (kind as above), w1, w2 decoded weights.
 * Writes G, U (may be NULL) and Y, each [nrows, N], for the listed rows. */
static int swiglu_rows_f64(const void *A, int kind, double sA,
                           const double *w1, const double *w2,
                           int64_t M, int64_t N, int64_t K,
                           const int64_t *rows, int64_t nrows,
                           double *G, double *U, double *Y)
{
    int bad = 0;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        if (m < 0 || m >= M)
            bad = 1;
    }
    if (bad)
        return -1;
#pragma omp parallel
    {
        double *a = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double *g = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        double *u = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows ? rows[i] : i;
            decode_a_row(A, kind, sA, m, K, a);
            gate_up_row(a, w1, w2, N, K, g, u);
            for (int64_t n = 0; n < N; ++n) {
                if (G)
                    G[i * N + n] = g[n];
                if (U)
                    U[i * N + n] = u[n];
                Y[i * N + n] = oracle_silu(g[n]) * u[n];
            }
        }
        free(a);
        free(g);
        free(u);
    }
    return 0;
}

/* Y = SiLU(A W1) * (A W2) for BF16 inputs given as raw 16-bit patterns.
 * A is [M,K], W1 and W2 are [K,N], all row-major.  G, U may be NULL.
 * Returns 0, or -1 on a bad row index / allocation failure. */
int oracle_swiglu_bf16(const uint16_t *A, const uint16_t *W1, const uint16_t *W2,
                       int64_t M, int64_t N, int64_t K,
                       const int64_t *rows, int64_t nrows,
                       double *G, double *U, double *Y)
{
    double *w1 = decode_bf16_matrix(W1, K * N);
    double *w2 = decode_bf16_matrix(W2, K * N);
    int rc = -1;
    if (w1 && w2)
        rc = swiglu_rows_f64(A, 0, 1.0, w1, w2, M, N, K, rows, nrows, G, U, Y);
    free(w1);
    free(w2);
    return rc;
}

/* FP8 E4M3 operands with per-tensor scales: every element is dequantised
 * (q * s, exact in double) and the same definition is applied. */
int oracle_swiglu_e4m3(const uint8_t *Aq, const uint8_t *W1q, const uint8_t *W2q,
                       double sA, double sW1, double sW2,
                       int64_t M, int64_t N, int64_t K,
                       const int64_t *rows, int64_t nrows,
                       double *G, double *U, double *Y)
{
    double *w1 = decode_e4m3_matrix(W1q, K * N, sW1);
    double *w2 = decode_e4m3_matrix(W2q, K * N, sW2);
    int rc = -1;
    if (w1 && w2)
        rc = swiglu_rows_f64(Aq, 1, sA, w1, w2, M, N, K, rows, nrows, G, U, Y);
    free(w1);
    free(w2);
    return rc;
}

/* ---- the interleaved form ("Kernel-2") --------------------------------- */

/* W_fused[k, 2n] = W1[k, n] (gate), W_fused[k, 2n+1] = W2[k, n] (up). */
void oracle_pack_interleaved_u16(const uint16_t *W1, const uint16_t *W2,
                                 uint16_t *Wf, int64_t K, int64_t N)
{
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            Wf[k * 2 * N + 2 * n] = W1[k * N + n];
            Wf[k * 2 * N + 2 * n + 1] = W2[k * N + n];
        }
}

void oracle_pack_interleaved_u8(const uint8_t *W1, const uint8_t *W2,
                                uint8_t *Wf, int64_t K, int64_t N)
{
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            Wf[k * 2 * N + 2 * n] = W1[k * N + n];
            Wf[k * 2 * N + 2 * n + 1] = W2[k * N + n];
        }
}

/* One GEMM D = A x W_fused over [M, 2N, K], then the pair step
 * Y[m,n] = SiLU(D[m,2n]) * D[m,2n+1], in the order the page gives. */
int oracle_swiglu_interleaved_bf16(const uint16_t *A, const uint16_t *Wf,
                                   int64_t M, int64_t N, int64_t K,
                                   const int64_t *rows, int64_t nrows,
                                   double *Y)
{
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        if (m < 0 || m >= M)
            return -1;
    }
    double *wf = decode_bf16_matrix(Wf, K * 2 * N);
    if (!wf)
        return -1;
    const int64_t N2 = 2 * N;
#pragma omp parallel
    {
        double *am = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double *d = (double *)malloc((size_t)(N2 > 0 ? N2 : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows ? rows[i] : i;
            decode_a_row(A, 0, 1.0, m, K, am);
            for (int64_t j = 0; j < N2; ++j)
                d[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double ak = am[k];
                const double *wk = wf + k * N2;
                for (int64_t j = 0; j < N2; ++j)
                    d[j] += ak * wk[j];
            }
            for (int64_t n = 0; n < N; ++n)
                Y[i * N + n] = oracle_silu(d[2 * n]) * d[2 * n + 1];
        }
        free(am);
        free(d);
    }
    free(wf);
    return 0;
}

/* ---- the next step of the MLP: the down projection ---------------------- */
/*
 * The page motivates the fused kernel by the MLP's total time (section
 * "Definizione del Problema": gate/up materialisation is 9-37 % of MLP time);
 * the MLP continues with a down projection Z = Y x W3 (+ residual R).  Between
 * the two projections Y is stored in BF16, as the fused kernel writes it, so
 * the MLP oracle rounds Y to BF16 once (round to nearest, ties to even) and
 * multiplies the rounded values exactly.
 */

/* Round a double to the nearest BF16 value, ties to even, returning the bit
 * pattern (no intermediate float rounding).  BF16: 1 sign, 8 exponent bits
 * (bias 127), 7 fraction bits; subnormals below 2^-126 have spacing 2^-133. */
uint16_t oracle_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    int e;
    frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    int q = e - 1;             /* a in [2^q, 2^(q+1)) */
    if (q < -126)
        q = -126;              /* subnormal range keeps the spacing of 2^-126's binade */
    double ulp = ldexp(1.0, q - 7);
    double m = nearbyint(a / ulp); /* exact division by a power of two; ties to even */
    double r = m * ulp;
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u); /* overflow to infinity */
    /* encode r */
    if (r < ldexp(1.0, -126)) {            /* subnormal: r = m * 2^-133 */
        return (uint16_t)(sign | (uint16_t)m);
    }
    int er;
    double fr = frexp(r, &er);             /* r = fr * 2^er, fr in [0.5, 1) */
    int biased = er - 1 + 127;
    uint16_t frac = (uint16_t)((fr * 2.0 - 1.0) * 128.0); /* exact: 7 fraction bits */
    return (uint16_t)(sign | (uint16_t)(biased << 7) | frac);
}

/* Z[r,:] = X[m_r,:] W (+ R[m_r,:]) in double, X [M,K], W [K,N], R [M,N] (may be NULL). */
int oracle_linear_bf16(const uint16_t *X, const uint16_t *W, const uint16_t *R,
                       int64_t M, int64_t N, int64_t K,
                       const int64_t *rows, int64_t nrows, double *Z)
{
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        if (m < 0 || m >= M)
            return -1;
    }
    double *w = decode_bf16_matrix(W, K * N);
    if (!w)
        return -1;
#pragma omp parallel
    {
        double *x = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double *z = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows ? rows[i] : i;
            decode_a_row(X, 0, 1.0, m, K, x);
            for (int64_t n = 0; n < N; ++n)
                z[n] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double xk = x[k];
                const double *wk = w + k * N;
                for (int64_t n = 0; n < N; ++n)
                    z[n] += xk * wk[n];
            }
            for (int64_t n = 0; n < N; ++n)
                Z[i * N + n] = z[n] + (R ? oracle_bf16_to_f64(R[m * N + n]) : 0.0);
        }
        free(x);
        free(z);
    }
    free(w);
    return 0;
}

/* The SwiGLU MLP block: Y = BF16(SiLU(A W1) (.) (A W2)) per row, then
 * Z = Y W3 (+ R).  A [M,H], W1/W2 [H,F], W3 [F,H], R [M,H] (may be NULL).
 * Writes Z [nrows,H] in double and, if Ybits is not NULL, the rounded Y
 * [nrows,F] as BF16 bit patterns. */
int oracle_mlp_bf16(const uint16_t *A, const uint16_t *W1, const uint16_t *W2,
                    const uint16_t *W3, const uint16_t *R,
                    int64_t M, int64_t H, int64_t F,
                    const int64_t *rows, int64_t nrows, double *Z, uint16_t *Ybits)
{
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        if (m < 0 || m >= M)
            return -1;
    }
    double *w1 = decode_bf16_matrix(W1, H * F);
    double *w2 = decode_bf16_matrix(W2, H * F);
    double *w3 = decode_bf16_matrix(W3, F * H);
    int rc = -1;
    if (w1 && w2 && w3) {
        rc = 0;
#pragma omp parallel
        {
            double *a = (double *)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
            double *g = (double *)malloc((size_t)(F > 0 ? F : 1) * sizeof(double));
            double *u = (double *)malloc((size_t)(F > 0 ? F : 1) * sizeof(double));
            double *y = (double *)malloc((size_t)(F > 0 ? F : 1) * sizeof(double));
            double *z = (double *)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < nrows; ++i) {
                int64_t m = rows ? rows[i] : i;
                decode_a_row(A, 0, 1.0, m, H, a);
                gate_up_row(a, w1, w2, F, H, g, u);
                for (int64_t f = 0; f < F; ++f) {
                    uint16_t yb = oracle_f64_to_bf16(oracle_silu(g[f]) * u[f]);
                    if (Ybits)
                        Ybits[i * F + f] = yb;
                    y[f] = oracle_bf16_to_f64(yb);
                }
                for (int64_t h = 0; h < H; ++h)
                    z[h] = 0.0;
                for (int64_t f = 0; f < F; ++f) {
                    const double yf = y[f];
                    const double *w3f = w3 + f * H;
                    for (int64_t h = 0; h < H; ++h)
                        z[h] += yf * w3f[h];
                }
                for (int64_t h = 0; h < H; ++h)
                    Z[i * H + h] = z[h] + (R ? oracle_bf16_to_f64(R[m * H + h]) : 0.0);
            }
            free(a);
            free(g);
            free(u);
            free(y);
            free(z);
        }
    }
    free(w1);
    free(w2);
    free(w3);
    return rc;
}

/* ---- the producer: RMSNorm and per-tensor FP8 quantisation of A --------
 *
 * The step that feeds the FP8 form of the projection.  The page names FP8
 * quantisation as what raises the tensor cores' arithmetic density (section
 * "Definizione del Problema") but defines neither the normalisation nor the
 * scaling, so these follow the plainest readings, listed in the design notes:
 *   - RMSNorm (root-mean-square layer normalisation, Zhang and Sennrich 2019):
 *     a[m,k] = x[m,k] * gamma[k] / sqrt(mean over k of x[m,k]^2 + eps); a row
 *     of zeros with eps = 0, where that is 0/0, normalises to zeros;
 *   - one scale for the whole tensor: s = max|a| / 448 (448 = the largest
 *     finite E4M3 value), rounded once to binary32 because the projection
 *     takes its scales as floats; s = 0 when every a is zero;
 *   - q = E4M3(a / s): the exact quotient of a and the binary32 scale,
 *     rounded to the nearest E4M3 value, ties to even, saturating at +-448,
 *     as the OCP 8-bit floating point specification defines conversion to
 *     E4M3 ("fn" variant); all codes are 0 when s = 0.  The quotient is taken
 *     in double, which resolves every decision the exact quotient makes
 *     except where it lies within 2^-53 of a midpoint.
 */

/* Round a double to FP8 E4M3 ("fn" variant, see oracle_e4m3_to_f64), ties to
 * even, clamping magnitudes beyond the finite range to 448.  Returns the bit
 * pattern.  Normal values in [2^q, 2^(q+1)) have spacing 2^(q-3); below 2^-6
 * the subnormals keep the spacing 2^-9 of the first binade. */
uint8_t oracle_f64_to_e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int e;
    frexp(a, &e);              /* a in [2^(e-1), 2^e) */
    int q = e - 1;
    if (q < -6)
        q = -6;
    double ulp = ldexp(1.0, q - 3);
    double m = nearbyint(a / ulp); /* exact division by a power of two; ties to even */
    double r = m * ulp;            /* a < 448 = 14 * 2^5, so r <= 448 */
    if (r < ldexp(1.0, -6))        /* subnormal: r = m * 2^-9, m in 0..7 */
        return (uint8_t)(sign | (uint8_t)m);
    int er;
    double fr = frexp(r, &er);     /* r = fr * 2^er, fr in [0.5, 1) */
    int biased = er - 1 + 7;
    uint8_t mant = (uint8_t)((fr * 2.0 - 1.0) * 8.0); /* exact: 3 fraction bits */
    return (uint8_t)(sign | (uint8_t)(biased << 3) | mant);
}

void oracle_f64_to_e4m3_n(const double *x, int64_t n, uint8_t *q)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = oracle_f64_to_e4m3(x[i]);
}

/* RMSNorm of every row of X [M,K] (BF16) in double; gamma [K] (BF16) may be
 * NULL, meaning all ones.  Writes A [M,K]. */
int oracle_rmsnorm_bf16(const uint16_t *X, const uint16_t *gamma, double eps,
                        int64_t M, int64_t K, double *A)
{
    if (M < 0 || K <= 0 || eps < 0.0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double x = oracle_bf16_to_f64(X[m * K + k]);
            ss += x * x;
        }
        double rms = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k) {
            double g = gamma ? oracle_bf16_to_f64(gamma[k]) : 1.0;
            A[m * K + k] = rms > 0.0 ? oracle_bf16_to_f64(X[m * K + k]) * g / rms : 0.0;
        }
    }
    return 0;
}

/* Per-tensor E4M3 quantisation of n values: *scale = (float)(max|a| / 448),
 * q[i] = E4M3(a[i] / scale), all zero when the scale is zero. */
int oracle_quant_e4m3(const double *a, int64_t n, float *scale, uint8_t *q)
{
    if (n < 0)
        return -1;
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double v = fabs(a[i]);
        if (isnan(v))
            return -1;
        if (v > amax)
            amax = v;
    }
    float s = (float)(amax / 448.0);
    *scale = s;
    for (int64_t i = 0; i < n; ++i)
        q[i] = s > 0.0f ? oracle_f64_to_e4m3(a[i] / (double)s) : 0;
    return 0;
}

/* ---- weight-only INT4 (a lower-precision weight variant) ----
 *
 * The page names INT4 as a precision that raises tensor-core density
 * (section "Definizione del Problema") without defining a format.  Reading
 * (the plainest common one): signed 4-bit weights q in [-8, 7], two's
 * complement, packed two per byte along N (byte k*(N/2) + n/2 holds column n
 * in its low nibble when n is even, in its high nibble when n is odd), one
 * BF16 scale per column and per group of G consecutive K rows; the weight the
 * product uses is the BF16 value of q * s (q * s is exact in binary32; it is
 * rounded once to BF16, nearest even), the form in which BF16 tensor cores
 * consume it.  Everything after that is the BF16 definition above.
 */
double oracle_int4_value(uint8_t nibble)
{
    int v = nibble & 0xF;
    return (double)(v < 8 ? v : v - 16);
}

/* W[k,n] = BF16(q[k,n] * S[k/G, n]) for Wq [K, N/2] bytes and S [K/G, N] BF16. */
int oracle_dequant_int4(const uint8_t *Wq, const uint16_t *S, int64_t K, int64_t N, int64_t G,
                        double *W)
{
    if (K < 0 || N < 0 || N % 2 != 0 || G <= 0 || K % G != 0)
        return -1;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            uint8_t byte = Wq[k * (N / 2) + n / 2];
            uint8_t nib = (n & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
            double p = oracle_int4_value(nib) * oracle_bf16_to_f64(S[(k / G) * N + n]);
            W[k * N + n] = oracle_bf16_to_f64(oracle_f64_to_bf16(p));
        }
    return 0;
}

/* The K-major arrangement of the same INT4 codes (a storage order only; the
 * values are unchanged): Wk [N, K/2] bytes, row n holding column n's codes;
 * 32-bit little-endian word j of a row holds codes k = 8j..8j+7, code 8j+2i
 * in nibble i and code 8j+2i+1 in nibble 4+i (i = 0..3), nibble p being bits
 * [4p, 4p+4) of the word, i.e. the low half of byte p/2 when p is even. */
int oracle_pack_w4_kmajor(const uint8_t *Wq, int64_t K, int64_t N, uint8_t *Wk)
{
    if (K < 0 || N < 0 || N % 2 != 0 || K % 8 != 0)
        return -1;
    for (int64_t i = 0; i < N * (K / 2); ++i)
        Wk[i] = 0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t code = (uint8_t)((Wq[k * (N / 2) + n / 2] >> (4 * (n % 2))) & 0xF);
            int64_t j = k / 8, r = k % 8;
            int64_t nib = (r % 2 == 0) ? r / 2 : 4 + r / 2;
            int64_t at = n * (K / 2) + 4 * j + nib / 2;
            Wk[at] |= (uint8_t)(code << (4 * (nib % 2)));
        }
    return 0;
}

/* Y = SiLU(A W1) (.) (A W2) with W1, W2 given as INT4 + group scales. */
int oracle_swiglu_w4(const uint16_t *A, const uint8_t *W1q, const uint16_t *S1,
                     const uint8_t *W2q, const uint16_t *S2, int64_t M, int64_t N, int64_t K,
                     int64_t G, const int64_t *rows, int64_t nrows, double *Y)
{
    double *w1 = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    double *w2 = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    int rc = -1;
    if (w1 && w2 && oracle_dequant_int4(W1q, S1, K, N, G, w1) == 0 &&
        oracle_dequant_int4(W2q, S2, K, N, G, w2) == 0)
        rc = swiglu_rows_f64(A, 0, 1.0, w1, w2, M, N, K, rows, nrows, NULL, NULL, Y);
    free(w1);
    free(w2);
    return rc;
}

/* ---- weight-only MXFP8 and NVFP4 (the block-scaled formats the GEMM page
 * names for Blackwell: "MXFP8" and "NVFP4" in its benchmark paragraph) ------
 *
 * Readings (the page names the formats only; these follow the published OCP
 * Microscaling specification and NVIDIA's NVFP4 description):
 *   MXFP8: E4M3 element codes (one byte each, row-major [K,N]); every block of
 *     32 consecutive K rows of a column shares one E8M0 scale (byte e: the
 *     value 2^(e - 127), e = 255 is NaN), scales [K/32, N].  Weight =
 *     BF16(E4M3(c) * 2^(e-127)) (exact unless the value leaves BF16's normal
 *     range).
 *   NVFP4: E2M1 element codes (1 sign, 2 exponent bits with bias 1, 1
 *     mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), packed two per
 *     byte along N like the INT4 codes; every block of 16 consecutive K rows
 *     of a column shares an E4M3 scale, scales [K/16, N]; one FP32 scale per
 *     tensor on top.  Weight = E2M1(c) * E4M3(s) * global.
 */
double oracle_e2m1_to_f64(uint8_t code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7];
    return (code & 8) ? -v : v;
}

double oracle_e8m0_to_f64(uint8_t e)
{
    if (e == 255)
        return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* W[k,n] = BF16(E4M3(C[k,n]) * E8M0(S[k/32, n])); C [K,N], S [K/32, N]. */
int oracle_dequant_mxfp8(const uint8_t *C, const uint8_t *S, int64_t K, int64_t N, double *W)
{
    if (K < 0 || N < 0 || K % 32 != 0)
        return -1;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            double v = oracle_e4m3_to_f64(C[k * N + n]) * oracle_e8m0_to_f64(S[(k / 32) * N + n]);
            W[k * N + n] = oracle_bf16_to_f64(oracle_f64_to_bf16(v));
        }
    return 0;
}

/* W[k,n] = E2M1(c[k,n]) * E4M3(S[k/16, n]) * global; C [K, N/2] packed. */
int oracle_dequant_nvfp4(const uint8_t *C, const uint8_t *S, double global, int64_t K, int64_t N,
                         double *W)
{
    if (K < 0 || N < 0 || N % 2 != 0 || K % 16 != 0)
        return -1;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            uint8_t byte = C[k * (N / 2) + n / 2];
            uint8_t code = (n & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
            W[k * N + n] = oracle_e2m1_to_f64(code) * oracle_e4m3_to_f64(S[(k / 16) * N + n]) * global;
        }
    return 0;
}

/* Y = SiLU(A W1) (.) (A W2) with MXFP8 (fmt 0) or NVFP4 (fmt 1) weights;
 * g1, g2: the NVFP4 per-tensor scales (ignored for MXFP8). */
int oracle_swiglu_mx(const uint16_t *A, int fmt, const uint8_t *C1, const uint8_t *S1, double g1,
                     const uint8_t *C2, const uint8_t *S2, double g2, int64_t M, int64_t N,
                     int64_t K, const int64_t *rows, int64_t nrows, double *Y)
{
    double *w1 = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    double *w2 = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    int rc = -1;
    if (w1 && w2) {
        int ok = fmt == 0 ? (oracle_dequant_mxfp8(C1, S1, K, N, w1) == 0 &&
                             oracle_dequant_mxfp8(C2, S2, K, N, w2) == 0)
                          : (oracle_dequant_nvfp4(C1, S1, g1, K, N, w1) == 0 &&
                             oracle_dequant_nvfp4(C2, S2, g2, K, N, w2) == 0);
        if (ok)
            rc = swiglu_rows_f64(A, 0, 1.0, w1, w2, M, N, K, rows, nrows, NULL, NULL, Y);
    }
    free(w1);
    free(w2);
    return rc;
}
