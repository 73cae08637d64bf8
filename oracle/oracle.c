/*
 * oracle.c -- plain fp64 CPU oracle for the fused pre-norm linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; the two meet only in the seeded inputs they are given.
 *
 * Every result here is the plain definition written out in double precision,
 * one row at a time, from the exact fp16/bf16 input values.  No blocking, no
 * fusion, no reordering beyond what the definitions state; the only liberty
 * taken is that independent output rows run on separate OpenMP threads.
 *
 * Sources (page title, then section):
 *  - "LayerNorm 融合算子如何让大模型推理再快 15%？深度拆解 ATB 的实现",
 *    §1.1 (LayerNorm in three steps: statistics, normalize, affine),
 *    §2.1 (the fused op is layer_norm followed by matmul with W transposed),
 *    §2.3 (statistics in FP32 -- here fp64), §6.2 (gamma folded into W in
 *    inference mode).
 *  - "昇腾CANN的MatMul融合玩法，让大模型推理快3倍", §二 strategy 1
 *    (MatMul + SiLU), strategy 2 (MatMul -> SiLU -> MatMul, the FFN),
 *    strategy 3 (RMSNorm + MatMul).
 *  - "CANN推理加速库ascend-transformer-boost ATB算子融合实战...", the
 *    LayerNormMatMul fusion section (fused_layernorm_matmul(x, w, bias));
 *    Llama2 inference, model structure and fusion opportunities (one
 *    RMSNorm feeding the Q/K/V projections; the FFN's SwiGLU, a SiLU-gated
 *    linear transform, fused with its matmuls).
 *  - "LayerNorm 融合算子如何让大模型推理再快 15%？", §3.3 (a fusion chain
 *    LayerNorm -> MatMul -> BiasAdd -> ReLU -> MatMul -> BiasAdd).
 *  - "昇腾CANN的MatMul融合玩法", the table of fused GEMM instructions
 *    (MatMul + ReLU / GELU / SiLU); §五 optimization 3 (the output
 *    projection fused with the RMSNorm that follows it).
 *
 * Readings taken where the pages are silent or at odds:
 *  - variance is the biased one (divide by K), as torch's layer_norm that
 *    §2.1 invokes; the §2.3 sketch's x.var() (unbiased) is read as a slip;
 *  - eps sits inside the square root for both LayerNorm and RMSNorm;
 *  - RMSNorm applies gamma, and no beta;
 *  - bias is optional; with SiLU the order is matmul, + bias, then SiLU;
 *  - SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z));
 *  - GELU(z) = z * Phi(z) = z (1 + erf(z / sqrt 2)) / 2, the exact form (the
 *    pages name GELU without defining it); ReLU(z) = max(z, 0);
 *  - SwiGLU is the Llama form h_j = SiLU(a . Wg[j]) * (a . Wu[j]) with the
 *    gate and up projections both [F, K] and no biases;
 *  - W is [N, K] row-major (the nn.Linear layout), y = a . W^T;
 *  - the FFN keeps its intermediate H in fp64, unrounded;
 *  - the post-product norm normalizes h = x . W^T + bias (+ residual) over
 *    its N columns, with gamma and beta of length N; the residual is
 *    optional (the page draws none; a transformer adds one there).
 *
 * Parity is pinned by tests from definitions, closed forms, invariants,
 * library routines in float64 and brute force on tiny inputs; the pages
 * print no worked numeric example for this path.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { NGO_F16 = 0, NGO_BF16 = 1 };
enum { NGO_NORM_NONE = 0, NGO_NORM_LAYER = 1, NGO_NORM_RMS = 2 };
enum { NGO_ACT_NONE = 0, NGO_ACT_SILU = 1, NGO_ACT_RELU = 2, NGO_ACT_GELU = 3 };

/* ---- exact decoding of the 16-bit inputs ---------------------------------
 * IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * bfloat16: the upper 16 bits of an IEEE-754 binary32.
 * Both convert to double exactly.  A 65536-entry table holds every value so
 * that each element is decoded by one lookup. */
static double decode_binary16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);    /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

static double decode_bfloat16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double g_table[2][65536];
static int g_table_ready[2];

static const double *table_for(int dt)
{
    if (!g_table_ready[dt]) {
        for (uint32_t i = 0; i < 65536u; ++i)
            g_table[dt][i] = dt == NGO_F16 ? decode_binary16((uint16_t)i)
                                           : decode_bfloat16((uint16_t)i);
        g_table_ready[dt] = 1;
    }
    return g_table[dt];
}

/* Decode n 16-bit values into doubles (exposed so tests can pin it). */
int ngo_decode(const uint16_t *src, int64_t n, int dt, double *dst)
{
    if (dt != NGO_F16 && dt != NGO_BF16) return -4;
    const double *T = table_for(dt);
    for (int64_t i = 0; i < n; ++i) dst[i] = T[src[i]];
    return 0;
}

/* ---- a1: row statistics ----------------------------------------------------
 * LayerNorm: mu = (1/K) sum_k x_k ; var = (1/K) sum_k (x_k - mu)^2 (two
 * passes, biased) ; rstd = 1 / sqrt(var + eps).
 * RMSNorm:   mu = 0 ; rstd = 1 / sqrt((1/K) sum_k x_k^2 + eps).
 * No norm:   mu = 0 ; rstd = 1. */
static void row_stats(int norm, const double *x, int64_t K, double eps,
                      double *mu_out, double *rstd_out)
{
    if (norm == NGO_NORM_LAYER) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += x[k];
        double mu = s / (double)K;
        double v = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double d = x[k] - mu;
            v += d * d;
        }
        v /= (double)K;
        *mu_out = mu;
        *rstd_out = 1.0 / sqrt(v + eps);
    } else if (norm == NGO_NORM_RMS) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += x[k] * x[k];
        *mu_out = 0.0;
        *rstd_out = 1.0 / sqrt(s / (double)K + eps);
    } else {
        *mu_out = 0.0;
        *rstd_out = 1.0;
    }
}

/* ---- a2: normalize + affine --------------------------------------------------
 * LayerNorm: a_k = (x_k - mu) * rstd * gamma_k + beta_k
 * RMSNorm:   a_k = x_k * rstd * gamma_k
 * No norm:   a_k = x_k */
static void normalize_row(int norm, const double *x, int64_t K, double mu,
                          double rstd, const double *gamma, const double *beta,
                          double *a)
{
    for (int64_t k = 0; k < K; ++k) {
        if (norm == NGO_NORM_LAYER)
            a[k] = (x[k] - mu) * rstd * gamma[k] + beta[k];
        else if (norm == NGO_NORM_RMS)
            a[k] = x[k] * rstd * gamma[k];
        else
            a[k] = x[k];
    }
}

/* SiLU(z) = z * sigmoid(z) */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* The activation applied after the bias. */
static double activation(int act, double z)
{
    switch (act) {
    case NGO_ACT_SILU: return silu(z);
    case NGO_ACT_RELU: return z > 0.0 ? z : 0.0;
    case NGO_ACT_GELU: return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
    default: return z;
    }
}

/* ---- a3 + a4: one output row of the linear layer -----------------------------
 * z_n = sum_k a_k * W[n, k] (+ bias_n) ; y_n = act(z_n).
 * W rows are decoded on the fly through the table. */
static void linear_row(const double *a, const uint16_t *W, const double *T,
                       const double *bias, int act, int64_t K, int64_t N,
                       double *y)
{
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t *w = W + n * K;
        double z = 0.0;
        for (int64_t k = 0; k < K; ++k) z += a[k] * T[w[k]];
        if (bias) z += bias[n];
        y[n] = activation(act, z);
    }
}

static int check_common(int dt, int64_t M, int64_t K, int64_t N,
                        const int64_t *rows, int64_t nrows)
{
    if (dt != NGO_F16 && dt != NGO_BF16) return -4;
    if (M < 0 || K <= 0 || N <= 0 || nrows < 0) return -2;
    if (rows)
        for (int64_t i = 0; i < nrows; ++i)
            if (rows[i] < 0 || rows[i] >= M) return -2;
    if (!rows && nrows > M) return -2;
    return 0;
}

/* Row statistics for the listed rows (all rows when rows == NULL). */
int ngo_row_stats(int norm, const uint16_t *x, int64_t M, int64_t K, int dt,
                  double eps, const int64_t *rows, int64_t nrows,
                  double *mu, double *rstd)
{
    int rc = check_common(dt, M, K, 1, rows, nrows);
    if (rc) return rc;
    const double *T = table_for(dt);
    int failed = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        if (!xr) { failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        row_stats(norm, xr, K, eps, &mu[i], &rstd[i]);
        free(xr);
    }
    return failed ? -9 : 0;
}

/* Normalized activations a[nrows, K] for the listed rows (step a2 alone). */
int ngo_normalize(int norm, const uint16_t *x, const uint16_t *gamma,
                  const uint16_t *beta, double eps, int64_t M, int64_t K,
                  int dt, const int64_t *rows, int64_t nrows, double *a)
{
    int rc = check_common(dt, M, K, 1, rows, nrows);
    if (rc) return rc;
    if (norm != NGO_NORM_NONE && !gamma) return -1;
    if (norm == NGO_NORM_LAYER && !beta) return -1;
    const double *T = table_for(dt);
    double *g = calloc((size_t)K, sizeof(double));
    double *b = calloc((size_t)K, sizeof(double));
    if (!g || !b) { free(g); free(b); return -9; }
    for (int64_t k = 0; k < K; ++k) {
        if (gamma) g[k] = T[gamma[k]];
        if (beta) b[k] = T[beta[k]];
    }
    int failed = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        if (!xr) { failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        double mu, rstd;
        row_stats(norm, xr, K, eps, &mu, &rstd);
        normalize_row(norm, xr, K, mu, rstd, g, b, a + i * K);
        free(xr);
    }
    free(g);
    free(b);
    return failed ? -9 : 0;
}

/* The fused layer for the listed rows: y[i, :] for row rows[i].
 * norm: none / LayerNorm / RMSNorm; act: none / SiLU; bias may be NULL. */
int ngo_norm_linear(int norm, int act, const uint16_t *x, const uint16_t *gamma,
                    const uint16_t *beta, const uint16_t *W,
                    const uint16_t *bias, double eps, int64_t M, int64_t K,
                    int64_t N, int dt, const int64_t *rows, int64_t nrows,
                    double *y)
{
    int rc = check_common(dt, M, K, N, rows, nrows);
    if (rc) return rc;
    if (!x || !W || !y) return -1;
    if (norm != NGO_NORM_NONE && !gamma) return -1;
    if (norm == NGO_NORM_LAYER && !beta) return -1;
    const double *T = table_for(dt);
    double *g = calloc((size_t)K, sizeof(double));
    double *b = calloc((size_t)K, sizeof(double));
    double *bi = bias ? calloc((size_t)N, sizeof(double)) : NULL;
    if (!g || !b || (bias && !bi)) { free(g); free(b); free(bi); return -9; }
    for (int64_t k = 0; k < K; ++k) {
        if (gamma) g[k] = T[gamma[k]];
        if (beta) b[k] = T[beta[k]];
    }
    if (bias)
        for (int64_t n = 0; n < N; ++n) bi[n] = T[bias[n]];
    int failed = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        double *a = malloc((size_t)K * sizeof(double));
        if (!xr || !a) { free(xr); free(a); failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        double mu, rstd;
        row_stats(norm, xr, K, eps, &mu, &rstd);
        normalize_row(norm, xr, K, mu, rstd, g, b, a);
        linear_row(a, W, T, bi, act, K, N, y + i * N);
        free(xr);
        free(a);
    }
    free(g);
    free(b);
    free(bi);
    return failed ? -9 : 0;
}

/* ---- a5: FFN chain -------------------------------------------------------------
 * h_j = SiLU(sum_k x_k * W1[j, k]) kept in fp64 ; y_n = sum_j h_j * W2[n, j]. */
int ngo_ffn(const uint16_t *x, const uint16_t *W1, const uint16_t *W2,
            int64_t M, int64_t K, int64_t F, int dt, const int64_t *rows,
            int64_t nrows, double *y)
{
    int rc = check_common(dt, M, K, F, rows, nrows);
    if (rc) return rc;
    if (!x || !W1 || !W2 || !y) return -1;
    const double *T = table_for(dt);
    int failed = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        double *h = malloc((size_t)F * sizeof(double));
        if (!xr || !h) { free(xr); free(h); failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        linear_row(xr, W1, T, NULL, NGO_ACT_SILU, K, F, h);
        linear_row(h, W2, T, NULL, NGO_ACT_NONE, F, K, y + i * K);
        free(xr);
        free(h);
    }
    return failed ? -9 : 0;
}

/* Decode a [n] 16-bit vector (NULL stays NULL); the caller frees. */
static double *decode_vec(const uint16_t *v, int64_t n, const double *T, int *failed)
{
    if (!v) return NULL;
    double *d = malloc((size_t)n * sizeof(double));
    if (!d) { *failed = 1; return NULL; }
    for (int64_t i = 0; i < n; ++i) d[i] = T[v[i]];
    return d;
}

/* ---- the general two-layer chain (LayerNorm fusion chain, FFN) ---------------
 * a = norm(x) ; h_j = act(a . W1[j] + b1_j) kept in fp64 ;
 * y_n = h . W2[n] + b2_n.  W1 is [F, K], W2 is [N, F]; b1, b2 may be NULL. */
int ngo_mlp(int norm, int act, const uint16_t *x, const uint16_t *gamma,
            const uint16_t *beta, const uint16_t *W1, const uint16_t *b1,
            const uint16_t *W2, const uint16_t *b2, double eps, int64_t M,
            int64_t K, int64_t F, int64_t N, int dt, const int64_t *rows,
            int64_t nrows, double *y)
{
    int rc = check_common(dt, M, K, F, rows, nrows);
    if (rc) return rc;
    if (N <= 0) return -2;
    if (!x || !W1 || !W2 || !y) return -1;
    if (norm != NGO_NORM_NONE && !gamma) return -1;
    if (norm == NGO_NORM_LAYER && !beta) return -1;
    const double *T = table_for(dt);
    int failed = 0;
    double *g = decode_vec(gamma, K, T, &failed);
    double *b = decode_vec(beta, K, T, &failed);
    double *c1 = decode_vec(b1, F, T, &failed);
    double *c2 = decode_vec(b2, N, T, &failed);
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        if (failed) continue;
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        double *a = malloc((size_t)K * sizeof(double));
        double *h = malloc((size_t)F * sizeof(double));
        if (!xr || !a || !h) { free(xr); free(a); free(h); failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        double mu, rstd;
        row_stats(norm, xr, K, eps, &mu, &rstd);
        normalize_row(norm, xr, K, mu, rstd, g, b, a);
        linear_row(a, W1, T, c1, act, K, F, h);
        linear_row(h, W2, T, c2, NGO_ACT_NONE, F, N, y + i * N);
        free(xr);
        free(a);
        free(h);
    }
    free(g);
    free(b);
    free(c1);
    free(c2);
    return failed ? -9 : 0;
}

/* ---- SwiGLU: one norm feeding the gate and up projections ---------------------
 * a = norm(x) ; h_j = SiLU(a . Wg[j]) * (a . Wu[j]) ; Wg, Wu are [F, K]. */
static void swiglu_row(const double *a, const uint16_t *Wg, const uint16_t *Wu,
                       const double *T, int64_t K, int64_t F, double *h)
{
    for (int64_t j = 0; j < F; ++j) {
        double zg = 0.0, zu = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            zg += a[k] * T[Wg[j * K + k]];
            zu += a[k] * T[Wu[j * K + k]];
        }
        h[j] = silu(zg) * zu;
    }
}

int ngo_swiglu(int norm, const uint16_t *x, const uint16_t *gamma, const uint16_t *beta,
               const uint16_t *Wg, const uint16_t *Wu, double eps, int64_t M,
               int64_t K, int64_t F, int dt, const int64_t *rows, int64_t nrows,
               double *h)
{
    int rc = check_common(dt, M, K, F, rows, nrows);
    if (rc) return rc;
    if (!x || !Wg || !Wu || !h) return -1;
    if (norm != NGO_NORM_NONE && !gamma) return -1;
    if (norm == NGO_NORM_LAYER && !beta) return -1;
    const double *T = table_for(dt);
    int failed = 0;
    double *g = decode_vec(gamma, K, T, &failed);
    double *b = decode_vec(beta, K, T, &failed);
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        if (failed) continue;
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        double *a = malloc((size_t)K * sizeof(double));
        if (!xr || !a) { free(xr); free(a); failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        double mu, rstd;
        row_stats(norm, xr, K, eps, &mu, &rstd);
        normalize_row(norm, xr, K, mu, rstd, g, b, a);
        swiglu_row(a, Wg, Wu, T, K, F, h + i * F);
        free(xr);
        free(a);
    }
    free(g);
    free(b);
    return failed ? -9 : 0;
}

/* The Llama MLP: h as ngo_swiglu (fp64, unrounded), y_n = h . Wd[n]; Wd is
 * [N, F]. */
int ngo_mlp_swiglu(int norm, const uint16_t *x, const uint16_t *gamma,
                   const uint16_t *beta, const uint16_t *Wg, const uint16_t *Wu,
                   const uint16_t *Wd, double eps, int64_t M, int64_t K, int64_t F,
                   int64_t N, int dt, const int64_t *rows, int64_t nrows, double *y)
{
    int rc = check_common(dt, M, K, F, rows, nrows);
    if (rc) return rc;
    if (N <= 0) return -2;
    if (!x || !Wg || !Wu || !Wd || !y) return -1;
    if (norm != NGO_NORM_NONE && !gamma) return -1;
    if (norm == NGO_NORM_LAYER && !beta) return -1;
    const double *T = table_for(dt);
    int failed = 0;
    double *g = decode_vec(gamma, K, T, &failed);
    double *b = decode_vec(beta, K, T, &failed);
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        if (failed) continue;
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        double *a = malloc((size_t)K * sizeof(double));
        double *h = malloc((size_t)F * sizeof(double));
        if (!xr || !a || !h) { free(xr); free(a); free(h); failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        double mu, rstd;
        row_stats(norm, xr, K, eps, &mu, &rstd);
        normalize_row(norm, xr, K, mu, rstd, g, b, a);
        swiglu_row(a, Wg, Wu, T, K, F, h);
        linear_row(h, Wd, T, NULL, NGO_ACT_NONE, F, N, y + i * N);
        free(xr);
        free(a);
        free(h);
    }
    free(g);
    free(b);
    return failed ? -9 : 0;
}

/* ---- a norm after the product ---------------------------------------------------
 * h_n = sum_k x_k W[n, k] + bias_n + residual_n ; y = norm(h) over n, i.e.
 * LayerNorm: (h_n - mu_h) rstd_h gamma_n + beta_n, RMSNorm: h_n rstd_h
 * gamma_n, with the statistics of the row h (two passes, fp64).  h is
 * returned too (unrounded).  bias and residual may be NULL. */
int ngo_linear_residual_norm(int norm, const uint16_t *x, const uint16_t *W,
                             const uint16_t *bias, const uint16_t *residual,
                             const uint16_t *gamma, const uint16_t *beta, double eps,
                             int64_t M, int64_t K, int64_t N, int dt,
                             const int64_t *rows, int64_t nrows, double *h, double *y)
{
    int rc = check_common(dt, M, K, N, rows, nrows);
    if (rc) return rc;
    if (norm != NGO_NORM_LAYER && norm != NGO_NORM_RMS) return -2;
    if (!x || !W || !gamma || !h || !y) return -1;
    if (norm == NGO_NORM_LAYER && !beta) return -1;
    const double *T = table_for(dt);
    int failed = 0;
    double *g = decode_vec(gamma, N, T, &failed);
    double *b = decode_vec(beta, N, T, &failed);
    double *bi = decode_vec(bias, N, T, &failed);
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        if (failed) continue;
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        if (!xr) { failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        double *hr = h + i * N;
        linear_row(xr, W, T, bi, NGO_ACT_NONE, K, N, hr);
        if (residual)
            for (int64_t n = 0; n < N; ++n) hr[n] += T[residual[r * N + n]];
        double mu, rstd;
        row_stats(norm, hr, N, eps, &mu, &rstd);
        normalize_row(norm, hr, N, mu, rstd, g, b, y + i * N);
        free(xr);
    }
    free(g);
    free(b);
    free(bi);
    return failed ? -9 : 0;
}

/* ---- a7: the inference-mode weight fold -----------------------------------------
 * "LayerNorm 融合算子如何让大模型推理再快 15%？", §6.2: in inference gamma and
 * beta are fixed, so gamma is folded into the matmul weight beforehand.
 * Written out:  a_k = (x_k - mu) rstd gamma_k + beta_k, so
 *   z_n = rstd * sum_k x_k (gamma_k W[n,k]) - rstd * mu * sum_k gamma_k W[n,k]
 *         + sum_k beta_k W[n,k] + bias_n
 * with W'[n,k] = gamma_k W[n,k], c_n = sum_k W'[n,k],
 * b'_n = sum_k beta_k W[n,k] + bias_n.  RMSNorm: mu = 0 and no beta term. */
int ngo_fold_prepare(int norm, const uint16_t *gamma, const uint16_t *beta,
                     const uint16_t *W, const uint16_t *bias, int64_t K,
                     int64_t N, int dt, double *Wf, double *c, double *bprime)
{
    if (dt != NGO_F16 && dt != NGO_BF16) return -4;
    if (norm != NGO_NORM_LAYER && norm != NGO_NORM_RMS) return -2;
    if (!gamma || !W || (norm == NGO_NORM_LAYER && !beta)) return -1;
    const double *T = table_for(dt);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double cn = 0.0, bn = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double w = T[W[n * K + k]];
            double wf = T[gamma[k]] * w;
            Wf[n * K + k] = wf;
            cn += wf;
            if (norm == NGO_NORM_LAYER) bn += T[beta[k]] * w;
        }
        c[n] = cn;
        bprime[n] = bn + (bias ? T[bias[n]] : 0.0);
    }
    return 0;
}

/* y_n = rstd * (x . W'[n]) - rstd * mu * c_n + b'_n, then the activation. */
int ngo_folded_linear(int norm, int act, const uint16_t *x, const double *Wf,
                      const double *c, const double *bprime, double eps,
                      int64_t M, int64_t K, int64_t N, int dt,
                      const int64_t *rows, int64_t nrows, double *y)
{
    int rc = check_common(dt, M, K, N, rows, nrows);
    if (rc) return rc;
    if (norm != NGO_NORM_LAYER && norm != NGO_NORM_RMS) return -2;
    const double *T = table_for(dt);
    int failed = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        double *xr = malloc((size_t)K * sizeof(double));
        if (!xr) { failed = 1; continue; }
        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[r * K + k]];
        double mu, rstd;
        row_stats(norm, xr, K, eps, &mu, &rstd);
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += xr[k] * Wf[n * K + k];
            double z = rstd * s - rstd * mu * c[n] + bprime[n];
            y[i * N + n] = activation(act, z);
        }
        free(xr);
    }
    return failed ? -9 : 0;
}

/* Number of OpenMP threads a parallel region here would use (1 without
 * OpenMP); reported beside CPU timings. */
int ngo_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
