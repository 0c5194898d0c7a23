/*
 * CPU oracle for row-wise RMSNorm and fused residual Add + RMSNorm, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain, fp64 statement of what the GPU
 * library computes. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the product path never does. It shares no code, header, table or helper
 * with the CUDA library, and it never reads a value produced by the CUDA library.
 *
 * What it follows.
 *   - The operation: the RMSNorm op listed among Machete's built-in ops ("Machete", section
 *     "Built-In Areas"), the "RMSNorm SM100" CuTe DSL example (CuTe DSL skill page, example
 *     index of "Workflow 0"), and KernelAgent-Oink's "RMSNorm and fused Add + RMSNorm" custom
 *     ops for SM100/SM103 (KernelAgent page, repository summary). None of the pages writes the
 *     formula out, so this file uses the standard definition of row-wise RMSNorm:
 *         r      = x + residual            (fused op only; plain op: r = x)
 *         rstd_i = 1 / sqrt( (1/N) sum_j r_ij^2 + eps )
 *         y_ij   = r_ij * rstd_i * w_j
 *   - The backward pass is the exact derivative of that definition (per row, with
 *     xhat = x * rstd and g = dy * w):
 *         dx_j = rstd * ( g_j - xhat_j * (1/N) sum_k g_k xhat_k )
 *         dw_j = sum over rows of dy_j * xhat_j
 *     which follows from d(rstd)/d(x_k) = -rstd^3 * x_k / N.
 *
 * Precision. Inputs arrive as raw bf16 bit patterns, fp32 or fp64 values; each element is
 * decoded exactly to fp64 and every step is done in fp64, in the order the definition reads
 * (sums run over j = 0..N-1 and over rows i = 0..M-1 in order). Outputs stay fp64: the
 * oracle never rounds to the GPU's storage type.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC oracle.c -lm (see libbuild.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element encodings accepted for every input tensor. */
enum { ORACLE_BF16 = 0, ORACLE_F32 = 1, ORACLE_F64 = 2 };

/* Return codes. */
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_NO_MEMORY = 2 };

/* A bf16 value is the upper 16 bits of an IEEE-754 binary32 value: widening it is exact. */
static double decode_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int valid_dtype(int dt) { return dt == ORACLE_BF16 || dt == ORACLE_F32 || dt == ORACLE_F64; }

/* Element `i` of a tensor stored with encoding `dt`, as an exact fp64 value. */
static double element(const void *base, int dt, int64_t i)
{
    if (dt == ORACLE_BF16) return decode_bf16(((const uint16_t *)base)[i]);
    if (dt == ORACLE_F32) return (double)((const float *)base)[i];
    return ((const double *)base)[i];
}

/* Decode n elements to fp64 (exposed so the tests can pin the decoding on its own). */
int oracle_decode(const void *src, int dt, int64_t n, double *dst)
{
    if (!src || !dst || n < 0 || !valid_dtype(dt)) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n; ++i) dst[i] = element(src, dt, i);
    return ORACLE_OK;
}

/* rstd = 1 / sqrt(mean(r^2) + eps) over one row r[0..N-1]. */
static double row_rstd(const double *r, int64_t N, double eps)
{
    double sum_sq = 0.0;
    for (int64_t j = 0; j < N; ++j) sum_sq += r[j] * r[j];
    double mean_sq = sum_sq / (double)N;
    return 1.0 / sqrt(mean_sq + eps);
}

/*
 * Fused residual Add + RMSNorm forward (KernelAgent page, repository summary: "fused Add +
 * RMSNorm"). `res` may be NULL, which gives the plain RMSNorm forward (Machete, "Built-In
 * Areas"). x, res: [M, N] row-major; w: [N]. Outputs (fp64, caller-owned, any may be NULL):
 * r_out [M, N] = x + res, y [M, N], rstd [M].
 */
int oracle_add_rmsnorm_fwd(const void *x, int x_dt, const void *res, int res_dt,
                           const void *w, int w_dt, int64_t M, int64_t N, double eps,
                           double *r_out, double *y, double *rstd)
{
    if (!x || !w || M < 0 || N < 1 || !valid_dtype(x_dt) || !valid_dtype(w_dt)) return ORACLE_BAD_ARG;
    if (res && !valid_dtype(res_dt)) return ORACLE_BAD_ARG;
    double *r = (double *)malloc((size_t)N * sizeof(double));
    double *wd = (double *)malloc((size_t)N * sizeof(double));
    if (!r || !wd) { free(r); free(wd); return ORACLE_NO_MEMORY; }
    for (int64_t j = 0; j < N; ++j) wd[j] = element(w, w_dt, j);

    for (int64_t i = 0; i < M; ++i) {
        /* r = x + residual (or x alone), exactly in fp64. */
        for (int64_t j = 0; j < N; ++j) {
            double v = element(x, x_dt, i * N + j);
            if (res) v += element(res, res_dt, i * N + j);
            r[j] = v;
        }
        double s = row_rstd(r, N, eps);
        if (rstd) rstd[i] = s;
        for (int64_t j = 0; j < N; ++j) {
            if (r_out) r_out[i * N + j] = r[j];
            if (y) y[i * N + j] = r[j] * s * wd[j];
        }
    }
    free(r);
    free(wd);
    return ORACLE_OK;
}

/* Plain RMSNorm forward: the fused op without a residual. */
int oracle_rmsnorm_fwd(const void *x, int x_dt, const void *w, int w_dt, int64_t M, int64_t N,
                       double eps, double *y, double *rstd)
{
    return oracle_add_rmsnorm_fwd(x, x_dt, NULL, 0, w, w_dt, M, N, eps, NULL, y, rstd);
}

/*
 * RMSNorm backward: the derivative of the forward definition above. rstd is recomputed in
 * fp64 from x and eps (the oracle takes nothing from a GPU forward pass).
 * dy, x: [M, N]; w: [N]. Outputs (fp64, caller-owned): dx [M, N] (may be NULL), dw [N]
 * (may be NULL; overwritten with the sum over all M rows, taken in row order).
 * It is the fused backward below with no gradient arriving at residual_out.
 */
/*
 * Fused residual Add + RMSNorm backward (the backward of the KernelAgent page's "fused Add +
 * RMSNorm", whose forward returns both y and residual_out = r = x + residual). Given the
 * gradient dy arriving at y and the gradient d_ro arriving at residual_out (may be NULL: zero),
 * the gradient with respect to r - and so with respect to both x and residual - is
 *     d_r = d_ro + (RMSNorm backward of dy at r)
 * and dw is the same as for the plain op. `r` is the forward's residual_out as stored.
 */
int oracle_add_rmsnorm_bwd(const void *dy, int dy_dt, const void *d_ro, int d_ro_dt,
                           const void *r, int r_dt, const void *w, int w_dt, int64_t M, int64_t N,
                           double eps, double *d_r, double *dw);

int oracle_rmsnorm_bwd(const void *dy, int dy_dt, const void *x, int x_dt, const void *w,
                       int w_dt, int64_t M, int64_t N, double eps, double *dx, double *dw)
{
    return oracle_add_rmsnorm_bwd(dy, dy_dt, NULL, 0, x, x_dt, w, w_dt, M, N, eps, dx, dw);
}

int oracle_add_rmsnorm_bwd(const void *dy, int dy_dt, const void *d_ro, int d_ro_dt,
                           const void *x, int x_dt, const void *w, int w_dt, int64_t M, int64_t N,
                           double eps, double *dx, double *dw)
{
    if (!dy || !x || !w || M < 0 || N < 1 || !valid_dtype(dy_dt) || !valid_dtype(x_dt) ||
        !valid_dtype(w_dt) || (d_ro && !valid_dtype(d_ro_dt)))
        return ORACLE_BAD_ARG;
    double *xr = (double *)malloc((size_t)N * sizeof(double));
    double *dyr = (double *)malloc((size_t)N * sizeof(double));
    double *wd = (double *)malloc((size_t)N * sizeof(double));
    double *xhat = (double *)malloc((size_t)N * sizeof(double));
    double *g = (double *)malloc((size_t)N * sizeof(double));
    if (!xr || !dyr || !wd || !xhat || !g) {
        free(xr); free(dyr); free(wd); free(xhat); free(g);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t j = 0; j < N; ++j) wd[j] = element(w, w_dt, j);
    if (dw)
        for (int64_t j = 0; j < N; ++j) dw[j] = 0.0;

    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            xr[j] = element(x, x_dt, i * N + j);
            dyr[j] = element(dy, dy_dt, i * N + j);
        }
        double s = row_rstd(xr, N, eps);
        double dot = 0.0; /* sum_k g_k * xhat_k */
        for (int64_t j = 0; j < N; ++j) {
            xhat[j] = xr[j] * s;
            g[j] = dyr[j] * wd[j];
            dot += g[j] * xhat[j];
        }
        double c = dot / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double grad = s * (g[j] - xhat[j] * c);
            if (d_ro) grad += element(d_ro, d_ro_dt, i * N + j);
            if (dx) dx[i * N + j] = grad;
            if (dw) dw[j] += dyr[j] * xhat[j];
        }
    }
    free(xr); free(dyr); free(wd); free(xhat); free(g);
    return ORACLE_OK;
}

/*
 * LayerNorm, the mean-subtracting variant of the same row norm (the CuTe DSL skill page lists a
 * "CTA norm (LayerNorm)" example in its "Workflow 0" example index). Standard definition, per
 * row of r = x (+ residual):
 *     mean = (1/N) sum_j r_j,   var = (1/N) sum_j (r_j - mean)^2,   rstd = 1 / sqrt(var + eps)
 *     y_j  = (r_j - mean) * rstd * w_j + b_j
 * `res` and `b` may be NULL (no residual, no bias). Outputs (fp64, any may be NULL): r_out,
 * y [M, N], mean [M], rstd [M].
 */
int oracle_add_layernorm_fwd(const void *x, int x_dt, const void *res, int res_dt, const void *w,
                             int w_dt, const void *b, int b_dt, int64_t M, int64_t N, double eps,
                             double *r_out, double *y, double *mean, double *rstd)
{
    if (!x || !w || M < 0 || N < 1 || !valid_dtype(x_dt) || !valid_dtype(w_dt) ||
        (res && !valid_dtype(res_dt)) || (b && !valid_dtype(b_dt)))
        return ORACLE_BAD_ARG;
    double *r = (double *)malloc((size_t)N * sizeof(double));
    double *wd = (double *)malloc((size_t)N * sizeof(double));
    double *bd = (double *)malloc((size_t)N * sizeof(double));
    if (!r || !wd || !bd) { free(r); free(wd); free(bd); return ORACLE_NO_MEMORY; }
    for (int64_t j = 0; j < N; ++j) {
        wd[j] = element(w, w_dt, j);
        bd[j] = b ? element(b, b_dt, j) : 0.0;
    }
    for (int64_t i = 0; i < M; ++i) {
        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double v = element(x, x_dt, i * N + j);
            if (res) v += element(res, res_dt, i * N + j);
            r[j] = v;
            sum += v;
        }
        double mu = sum / (double)N;
        double sq = 0.0;
        for (int64_t j = 0; j < N; ++j) sq += (r[j] - mu) * (r[j] - mu);
        double s = 1.0 / sqrt(sq / (double)N + eps);
        if (mean) mean[i] = mu;
        if (rstd) rstd[i] = s;
        for (int64_t j = 0; j < N; ++j) {
            if (r_out) r_out[i * N + j] = r[j];
            if (y) y[i * N + j] = (r[j] - mu) * s * wd[j] + bd[j];
        }
    }
    free(r); free(wd); free(bd);
    return ORACLE_OK;
}

/*
 * LayerNorm backward (the exact derivative of the definition above), with xhat = (x - mean) *
 * rstd and g = dy * w, per row:
 *     dx_j = rstd * ( g_j - mean_k(g_k) - xhat_j * mean_k(g_k * xhat_k) )  (+ d_ro_j, fused)
 *     dw_j = sum over rows of dy_j * xhat_j,   db_j = sum over rows of dy_j
 * mean and rstd are recomputed in fp64 from x (the stored residual_out for the fused op).
 * d_ro may be NULL. Outputs (fp64, any may be NULL): dx [M, N], dw [N], db [N].
 */
int oracle_add_layernorm_bwd(const void *dy, int dy_dt, const void *d_ro, int d_ro_dt,
                             const void *x, int x_dt, const void *w, int w_dt, int64_t M,
                             int64_t N, double eps, double *dx, double *dw, double *db)
{
    if (!dy || !x || !w || M < 0 || N < 1 || !valid_dtype(dy_dt) || !valid_dtype(x_dt) ||
        !valid_dtype(w_dt) || (d_ro && !valid_dtype(d_ro_dt)))
        return ORACLE_BAD_ARG;
    double *xr = (double *)malloc((size_t)N * sizeof(double));
    double *dyr = (double *)malloc((size_t)N * sizeof(double));
    double *wd = (double *)malloc((size_t)N * sizeof(double));
    double *xhat = (double *)malloc((size_t)N * sizeof(double));
    double *g = (double *)malloc((size_t)N * sizeof(double));
    if (!xr || !dyr || !wd || !xhat || !g) {
        free(xr); free(dyr); free(wd); free(xhat); free(g);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t j = 0; j < N; ++j) wd[j] = element(w, w_dt, j);
    if (dw) for (int64_t j = 0; j < N; ++j) dw[j] = 0.0;
    if (db) for (int64_t j = 0; j < N; ++j) db[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            xr[j] = element(x, x_dt, i * N + j);
            dyr[j] = element(dy, dy_dt, i * N + j);
            sum += xr[j];
        }
        double mu = sum / (double)N;
        double sq = 0.0;
        for (int64_t j = 0; j < N; ++j) sq += (xr[j] - mu) * (xr[j] - mu);
        double s = 1.0 / sqrt(sq / (double)N + eps);
        double sum_g = 0.0, sum_gx = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            xhat[j] = (xr[j] - mu) * s;
            g[j] = dyr[j] * wd[j];
            sum_g += g[j];
            sum_gx += g[j] * xhat[j];
        }
        double mg = sum_g / (double)N, mgx = sum_gx / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double grad = s * (g[j] - mg - xhat[j] * mgx);
            if (d_ro) grad += element(d_ro, d_ro_dt, i * N + j);
            if (dx) dx[i * N + j] = grad;
            if (dw) dw[j] += dyr[j] * xhat[j];
            if (db) db[j] += dyr[j];
        }
    }
    free(xr); free(dyr); free(wd); free(xhat); free(g);
    return ORACLE_OK;
}

/*
 * FP8 E4M3 (the "e4m3fn" encoding: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, 0x7F/0xFF are NaN, largest finite 448). Decoding is exact; encoding rounds to
 * nearest, ties to even, and saturates finite values beyond 448 to +/-448 (the "satfinite"
 * conversion a quantising kernel uses). Written from the format's definition.
 */
double oracle_e4m3_decode(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
    if (e == 0xF && m == 7) return NAN;
    double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

uint8_t oracle_e4m3_encode(double v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E;
    /* The 127 non-negative finite codes are ordered by value: take the nearest, ties to the
     * even code (the one whose last mantissa bit is 0). */
    uint8_t best = 0;
    for (uint8_t c = 1; c <= 0x7E; ++c) {
        double dc = oracle_e4m3_decode(c), db = oracle_e4m3_decode(best);
        double ec = fabs(dc - a), eb = fabs(db - a);
        if (ec < eb || (ec == eb && (c & 1) == 0)) best = c;
    }
    return sign | best;
}

/*
 * RMSNorm (fused with the residual add when `res` is not NULL) feeding an FP8 E4M3 output with
 * one scale per row - the fusion with the neighbouring op that a persistent megakernel would do
 * (Machete, "Core Ideas": one instruction stream across ops). Per row:
 *     y = r * rstd * w                         (as oracle_add_rmsnorm_fwd)
 *     amax = max_j |y_j|;  scale = amax / 448  (scale = 0 for an all-zero y)
 *     v_j = y_j / scale (0 when scale = 0);    q_j = e4m3(v_j)
 * Outputs (any may be NULL): r_out, v [M, N] (the real-valued code target, fp64),
 * q [M, N] (the codes, taking the rounding decision on v), scale [M], rstd [M].
 */
int oracle_rmsnorm_quant_fp8(const void *x, int x_dt, const void *res, int res_dt, const void *w,
                             int w_dt, int64_t M, int64_t N, double eps, double *r_out, double *v,
                             uint8_t *q, double *scale, double *rstd)
{
    if (!x || !w || M < 0 || N < 1) return ORACLE_BAD_ARG;
    double *y = (double *)malloc((size_t)N * sizeof(double));
    double *rr = (double *)malloc((size_t)N * sizeof(double));
    double *s = (double *)malloc(sizeof(double));
    if (!y || !rr || !s) { free(y); free(rr); free(s); return ORACLE_NO_MEMORY; }
    int st = ORACLE_OK;
    for (int64_t i = 0; i < M && st == ORACLE_OK; ++i) {
        /* one row through the plain definition above */
        const char *xb = (const char *)x, *rb = (const char *)res;
        int xs = x_dt == ORACLE_BF16 ? 2 : x_dt == ORACLE_F32 ? 4 : 8;
        int rs = res_dt == ORACLE_BF16 ? 2 : res_dt == ORACLE_F32 ? 4 : 8;
        st = oracle_add_rmsnorm_fwd(xb + (size_t)(i * N) * xs, x_dt,
                                    res ? rb + (size_t)(i * N) * rs : NULL, res_dt, w, w_dt, 1, N,
                                    eps, rr, y, s);
        if (st != ORACLE_OK) break;
        double amax = 0.0;
        for (int64_t j = 0; j < N; ++j) amax = fmax(amax, fabs(y[j]));
        double sc = amax / 448.0;
        if (scale) scale[i] = sc;
        if (rstd) rstd[i] = *s;
        for (int64_t j = 0; j < N; ++j) {
            double vv = sc > 0.0 ? y[j] / sc : 0.0;
            if (r_out) r_out[i * N + j] = rr[j];
            if (v) v[i * N + j] = vv;
            if (q) q[i * N + j] = oracle_e4m3_encode(vv);
        }
    }
    free(y); free(rr); free(s);
    return st;
}
