/*
 * oracle.c -- plain, slow, fp64 CPU reference for the epilogue-fusion hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it (through oracle/__init__.py).  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Sources (page title, section):
 *   "Fusing an Epilogue" (docs.teenygrad.org, kernels/patterns/fusion),
 *     "The problem" (conv -> batchnorm -> silu chain),
 *     "The shape of it" (epilogue pseudocode: acc*bn_scale + bn_bias, then
 *     acc*sigmoid(acc)),
 *     the BatchNorm-epilog listing (one scale and one bias per output channel).
 *   "When the fusion you want is impossible, fuse into the producer"
 *     (skandtandon.pages.dev), last section: filters stored channels-last
 *     once at load time, bit-identical output.
 *   "Costs and benefits of kernel fusion" (intro-to-ai-systems-performance),
 *     opening example y = GELU(x + bias) over 67M fp16 values, and
 *     "Worked example: Fusing a residual and normalization chain".
 *
 * Everything is computed in double precision from the exact values of the
 * bf16 / fp16 / fp32 inputs.  Loops follow the plain definitions; the only
 * parallelism is a split of independent outputs over POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- storage formats, decoded from their IEEE definitions ------------- */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);    /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 value, ties to even, and return it
 * as a double.  Used only where the unfused chain materialises an fp16
 * intermediate. */
static double round_to_f16(double v)
{
    if (v != v || isinf(v))
        return v;
    double a = fabs(v);
    if (a >= 65520.0)                      /* rounds past the largest finite */
        return v < 0 ? -INFINITY : INFINITY;
    int e;
    frexp(a, &e);                          /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 11;                        /* spacing 2^q for 11 significant bits */
    if (q < -24)
        q = -24;                           /* subnormal spacing */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);   /* default mode: ties to even */
    return v < 0 ? -r : r;
}

/* Same for bfloat16 (8 significant bits, binary32 exponent range). */
static double round_to_bf16(double v)
{
    if (v != v || isinf(v))
        return v;
    double a = fabs(v);
    if (a == 0.0)
        return v;
    int e;
    frexp(a, &e);
    int q = e - 8;
    if (q < -133)
        q = -133;                          /* subnormal spacing: 2^-126 with 7 fraction bits */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r > 3.3895313892515355e38)
        r = INFINITY;
    return v < 0 ? -r : r;
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* ---- thread split over independent outputs ---------------------------- */

typedef void (*range_fn)(void *ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void *ctx; int64_t lo, hi; } range_job;

static void *run_range(void *p)
{
    range_job *j = (range_job *)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > n)
        nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[256];
    range_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = n * t / nthreads;
        jobs[t].hi = n * (t + 1) / nthreads;
        pthread_create(&th[t], NULL, run_range, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_join(th[t], NULL);
}

/* ---- filter layout change -------------------------------------------- */

/* "fuse into the producer", last section: store the filters channels-last
 * once, at load time.  w_oihw is [C_out][C_in][KH][KW]; w_ohwi is
 * [C_out][KH][KW][C_in].  A pure permutation of the 16-bit words. */
void oracle_pack_filter(const uint16_t *w_oihw, uint16_t *w_ohwi,
                        int C_out, int C_in, int KH, int KW)
{
    for (int co = 0; co < C_out; ++co)
        for (int ci = 0; ci < C_in; ++ci)
            for (int kh = 0; kh < KH; ++kh)
                for (int kw = 0; kw < KW; ++kw)
                    w_ohwi[(((int64_t)co * KH + kh) * KW + kw) * C_in + ci] =
                        w_oihw[(((int64_t)co * C_in + ci) * KH + kh) * KW + kw];
}

/* ---- conv2d + BatchNorm(scale, bias) + SiLU ---------------------------- */

enum { EPI_NONE = 0, EPI_FUSED = 1, EPI_CHAIN = 2 };

typedef struct {
    const uint16_t *x;       /* NHWC bf16 */
    const uint16_t *w;       /* OIHW bf16 (read directly: no pack involved) */
    const float *scale, *bias;
    int N, H, W, Ci, Co, KH, KW, sh, sw, ph, pw, Ho, Wo;
    int epilogue;
    const int64_t *points;   /* NULL: every output; else flat NHWC output indices */
    double *y;
} conv_ctx;

/* One output element y[n][oh][ow][co]:
 *   acc = sum over kh, kw, ci of x[n][oh*sh-ph+kh][ow*sw-pw+kw][ci] * w[co][ci][kh][kw]
 *         (taps that fall outside the input read zero),
 *   then the epilogue of "The shape of it": acc*bn_scale + bn_bias, then
 *   value * sigmoid(value).
 * EPI_CHAIN rounds to bf16 where the three-operation chain of "The problem"
 * writes t1 and t2 to memory. */
static double conv_point(const conv_ctx *c, int n, int oh, int ow, int co)
{
    double acc = 0.0;
    for (int kh = 0; kh < c->KH; ++kh) {
        int ih = oh * c->sh - c->ph + kh;
        if (ih < 0 || ih >= c->H)
            continue;
        for (int kw = 0; kw < c->KW; ++kw) {
            int iw = ow * c->sw - c->pw + kw;
            if (iw < 0 || iw >= c->W)
                continue;
            const uint16_t *xp = c->x + (((int64_t)n * c->H + ih) * c->W + iw) * c->Ci;
            for (int ci = 0; ci < c->Ci; ++ci) {
                double wv = bf16_value(c->w[(((int64_t)co * c->Ci + ci) * c->KH + kh) * c->KW + kw]);
                acc += bf16_value(xp[ci]) * wv;
            }
        }
    }
    if (c->epilogue == EPI_NONE)
        return acc;
    if (c->epilogue == EPI_CHAIN) {
        double t1 = round_to_bf16(acc);
        double t2 = round_to_bf16(t1 * (double)c->scale[co] + (double)c->bias[co]);
        return t2 * sigmoid(t2);
    }
    double v = acc * (double)c->scale[co] + (double)c->bias[co];
    return v * sigmoid(v);
}

static void conv_range(void *p, int64_t lo, int64_t hi)
{
    const conv_ctx *c = (const conv_ctx *)p;
    for (int64_t i = lo; i < hi; ++i) {
        int64_t flat = c->points ? c->points[i] : i;
        int64_t r = flat;
        int co = (int)(r % c->Co); r /= c->Co;
        int ow = (int)(r % c->Wo); r /= c->Wo;
        int oh = (int)(r % c->Ho); r /= c->Ho;
        int n = (int)r;
        c->y[i] = conv_point(c, n, oh, ow, co);
    }
}

/* Output spatial size of a convolution: floor((H + 2p - K) / s) + 1. */
static int out_dim(int H, int K, int s, int p) { return (H + 2 * p - K) / s + 1; }

/* Every output element, y in NHWC [N][Ho][Wo][C_out]. */
void oracle_conv2d_bn_silu(const uint16_t *x, const uint16_t *w_oihw,
                           const float *scale, const float *bias,
                           int N, int H, int W, int C_in, int C_out, int KH, int KW,
                           int sh, int sw, int ph, int pw, int epilogue,
                           double *y, int nthreads)
{
    conv_ctx c = {x, w_oihw, scale, bias, N, H, W, C_in, C_out, KH, KW, sh, sw, ph, pw,
                  out_dim(H, KH, sh, ph), out_dim(W, KW, sw, pw), epilogue, NULL, y};
    int64_t total = (int64_t)N * c.Ho * c.Wo * C_out;
    parallel_for(total, nthreads, conv_range, &c);
}

/* Selected output elements, by flat NHWC index into [N][Ho][Wo][C_out]. */
void oracle_conv2d_bn_silu_points(const uint16_t *x, const uint16_t *w_oihw,
                                  const float *scale, const float *bias,
                                  int N, int H, int W, int C_in, int C_out, int KH, int KW,
                                  int sh, int sw, int ph, int pw, int epilogue,
                                  const int64_t *points, int64_t npoints,
                                  double *y, int nthreads)
{
    conv_ctx c = {x, w_oihw, scale, bias, N, H, W, C_in, C_out, KH, KW, sh, sw, ph, pw,
                  out_dim(H, KH, sh, ph), out_dim(W, KW, sw, pw), epilogue, points, y};
    parallel_for(npoints, nthreads, conv_range, &c);
}

/* ---- y = GELU(x + bias) ------------------------------------------------ */

typedef struct {
    const uint16_t *x, *bias;   /* fp16 [rows][cols], fp16 [cols] */
    int64_t rows, cols;
    int materialize;
    double *y;
    double *rowsum;             /* optional: sum over each row of y */
} gelu_ctx;

/* GELU with the erf definition, s * Phi(s), Phi the standard normal CDF,
 * written as 0.5 * s * erfc(-s / sqrt(2)) so that the negative tail keeps
 * its relative accuracy.  "Costs and benefits of kernel fusion", opening
 * example.  With materialize set, x + bias is first rounded to fp16, as the
 * eager two-kernel version stores it. */
static double gelu_of_sum(double s) { return 0.5 * s * erfc(-s / sqrt(2.0)); }

static void gelu_range(void *p, int64_t lo, int64_t hi)
{
    const gelu_ctx *c = (const gelu_ctx *)p;
    for (int64_t r = lo; r < hi; ++r) {
        double acc = 0.0;
        for (int64_t j = 0; j < c->cols; ++j) {
            double s = f16_value(c->x[r * c->cols + j]) + f16_value(c->bias[j]);
            if (c->materialize)
                s = round_to_f16(s);
            double g = gelu_of_sum(s);
            if (c->y)
                c->y[r * c->cols + j] = g;
            acc += g;
        }
        if (c->rowsum)
            c->rowsum[r] = acc;
    }
}

void oracle_bias_gelu(const uint16_t *x, const uint16_t *bias, int64_t rows, int64_t cols,
                      int materialize, double *y, int nthreads)
{
    gelu_ctx c = {x, bias, rows, cols, materialize, y, NULL};
    parallel_for(rows, nthreads, gelu_range, &c);
}

/* The exercise at the end of "Costs and benefits of kernel fusion": bias,
 * GELU and a per-row reduction (the sum of each row of GELU(x + bias)). */
void oracle_bias_gelu_rowsum(const uint16_t *x, const uint16_t *bias, int64_t rows, int64_t cols,
                             int materialize, double *y, double *rowsum, int nthreads)
{
    gelu_ctx c = {x, bias, rows, cols, materialize, y, rowsum};
    parallel_for(rows, nthreads, gelu_range, &c);
}

/* ---- residual + LayerNorm + affine ------------------------------------- */

typedef struct {
    const uint16_t *act, *res;     /* fp16 [rows][hidden] */
    const float *gamma, *beta;     /* fp32 [hidden] */
    int64_t rows, hidden;
    double eps;
    int materialize;
    double *y;
    double *stats;                 /* optional [rows][2]: mean, variance */
} ln_ctx;

/* "Worked example: Fusing a residual and normalization chain": s = act + res;
 * row statistics mean = sum(s)/H and variance = sum((s-mean)^2)/H (two
 * passes, biased estimator); (s - mean)/sqrt(variance + eps); then scale by
 * gamma and add beta.  With materialize set, s and the normalised row are
 * rounded to fp16 where the eager three-kernel graph writes them. */
static void ln_range(void *p, int64_t lo, int64_t hi)
{
    const ln_ctx *c = (const ln_ctx *)p;
    int64_t H = c->hidden;
    double *s = (double *)malloc(sizeof(double) * (size_t)H);
    for (int64_t r = lo; r < hi; ++r) {
        for (int64_t j = 0; j < H; ++j) {
            double v = f16_value(c->act[r * H + j]) + f16_value(c->res[r * H + j]);
            s[j] = c->materialize ? round_to_f16(v) : v;
        }
        double sum = 0.0;
        for (int64_t j = 0; j < H; ++j)
            sum += s[j];
        double mean = sum / (double)H;
        double sq = 0.0;
        for (int64_t j = 0; j < H; ++j)
            sq += (s[j] - mean) * (s[j] - mean);
        double var = sq / (double)H;
        double inv = 1.0 / sqrt(var + c->eps);
        for (int64_t j = 0; j < H; ++j) {
            double nrm = (s[j] - mean) * inv;
            if (c->materialize)
                nrm = round_to_f16(nrm);
            c->y[r * H + j] = nrm * (double)c->gamma[j] + (double)c->beta[j];
        }
        if (c->stats) {
            c->stats[2 * r] = mean;
            c->stats[2 * r + 1] = var;
        }
    }
    free(s);
}

void oracle_residual_layernorm(const uint16_t *act, const uint16_t *res,
                               const float *gamma, const float *beta,
                               int64_t rows, int64_t hidden, double eps, int materialize,
                               double *y, double *stats, int nthreads)
{
    ln_ctx c = {act, res, gamma, beta, rows, hidden, eps, materialize, y, stats};
    parallel_for(rows, nthreads, ln_range, &c);
}

/* ---- exported scalar helpers (used by the oracle's own tests) ---------- */

double oracle_f16_value(uint16_t h) { return f16_value(h); }
double oracle_bf16_value(uint16_t b) { return bf16_value(b); }
double oracle_round_to_f16(double v) { return round_to_f16(v); }
double oracle_round_to_bf16(double v) { return round_to_bf16(v); }
double oracle_gelu(double s) { return gelu_of_sum(s); }
double oracle_silu(double v) { return v * sigmoid(v); }
