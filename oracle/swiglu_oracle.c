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
