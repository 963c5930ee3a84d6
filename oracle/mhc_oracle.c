/*
 * mhc_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, obviously-correct CPU statement of the manifold-constrained
 * hyper-connection (mHC) seam: the delayed pre block and the post block.
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
 * load this file's library.  It shares no code, header or constant with the
 * CUDA path.
 *
 * Sources (vLLM pull requests, as quoted on the web pages this work follows):
 *  - "[ROCm][DSV4.1][Perf] Use AITER mHC for the delayed pre block" (#56503),
 *    commit message and sections "Why V4.1 cannot just reuse MHCPreOp",
 *    "Approach", "Result", "Notes / follow-ups": the delayed pre collapses a
 *    sublayer's input with the previous seam's pre-mix and returns its own;
 *    the projection with each row's sum of squares; the post and comb gates;
 *    20 Sinkhorn iterations on a 4x4 comb; the collapse is a plain fp32
 *    weighted sum, bit-exact between implementations.
 *  - "[ROCm][DSv4.1] Fix TileLang mHC pre on 64-wide wavefronts ..." (#56342),
 *    sections "The bug" and "Measurements": the fused RMSNorm fold computes
 *    x * rsqrt * norm_weight in fp32 and rounds once.
 *  The pages print none of the gate or Sinkhorn formulas; the readings taken
 *  where they are silent are listed beside each function below.
 *
 * Arithmetic: everything in fp64 except the collapse, which also has the
 * exact fp32 path (each product rounded to fp32, sums left to right in stream
 * order, no fused multiply-add -- build with -ffp-contract=off) because the
 * pages state that the collapse is bit-exact between implementations.
 *
 * Parity pins: every function here is pinned by the CPU tests (closed forms,
 * invariants, a 50-digit brute force at T=1, C=8, library cross-checks).
 * Whether the gate/Sinkhorn readings match the production model the pages
 * describe is not pinned (parity unpinned against that model: no code or
 * weights of it are available); the readings define the method here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 bit pattern -> exact value. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an exact double to the nearest bf16 (ties to even), one rounding.
 * bf16: 1 sign bit, 8 exponent bits (same range as fp32), 8 significant bits.
 * The grid spacing at |v| in [2^(e-1), 2^e) is 2^(e-8); below the normal
 * range it is the subnormal step 2^-133. */
static uint16_t bf16_round(double v)
{
    if (isnan(v))
        return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (a >= 0x1p128)
        return sign | 0x7f80;
    int e;
    frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
    int step = e - 8;
    if (step < -133)
        step = -133;
    double q = nearbyint(ldexp(a, -step)); /* default mode: nearest, ties even */
    double r = ldexp(q, step);
    if (r >= 0x1p128)
        return sign | 0x7f80;
    float f = (float)r;      /* exact: r is on the bf16 grid */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7fff);
}

ORACLE_API void mhc_oracle_bf16_round(const double *v, int64_t count, uint16_t *out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = bf16_round(v[i]);
}

/* ----------------------------------------------------------- Sinkhorn --- */

/* Comb matrix from the n*n comb logits, row-major: comb[i][j] comes from
 * logit (2n + i*n + j); row i is the source stream, column j the destination.
 *
 * Readings (the pages give "20 Sinkhorn iterations" on the 4x4 comb and an
 * eager census of one softmax plus 39 sums per seam):
 *  - iteration 1: row-wise softmax (max subtracted per row), then eps added
 *    to every entry once, then column normalisation;
 *  - iterations 2..iters: row normalisation, then column normalisation;
 *  - no eps in any denominator. */
static void sinkhorn(const double *l, int n, int iters, double eps, double *P)
{
    for (int i = 0; i < n; ++i) {
        double mx = l[i * n];
        for (int j = 1; j < n; ++j)
            if (l[i * n + j] > mx)
                mx = l[i * n + j];
        double s = 0.0;
        for (int j = 0; j < n; ++j) {
            P[i * n + j] = exp(l[i * n + j] - mx);
            s += P[i * n + j];
        }
        for (int j = 0; j < n; ++j)
            P[i * n + j] = P[i * n + j] / s + eps;
    }
    for (int it = 0; it < iters; ++it) {
        if (it > 0) {
            for (int i = 0; i < n; ++i) {
                double s = 0.0;
                for (int j = 0; j < n; ++j)
                    s += P[i * n + j];
                for (int j = 0; j < n; ++j)
                    P[i * n + j] /= s;
            }
        }
        for (int j = 0; j < n; ++j) {
            double s = 0.0;
            for (int i = 0; i < n; ++i)
                s += P[i * n + j];
            for (int i = 0; i < n; ++i)
                P[i * n + j] /= s;
        }
    }
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Gates and comb from one token's 2n+n^2 logits:
 * pre = sigmoid(l[0:n]), post = 2*sigmoid(l[n:2n]), comb = Sinkhorn(l[2n:]). */
static void gates_from_logits(const double *l, int n, int iters, double eps,
                              double *pre, double *post, double *comb)
{
    for (int i = 0; i < n; ++i) {
        pre[i] = sigmoid(l[i]);
        post[i] = 2.0 * sigmoid(l[n + i]);
    }
    sinkhorn(l + 2 * n, n, iters, eps, comb);
}

ORACLE_API int mhc_oracle_gates_from_logits(const double *logits, int64_t T, int n,
                                            int iters, double sinkhorn_eps,
                                            double *pre, double *post, double *comb)
{
    if (n < 1 || iters < 1 || T < 0)
        return 1;
    const int M = 2 * n + n * n;
    for (int64_t t = 0; t < T; ++t)
        gates_from_logits(logits + t * M, n, iters, sinkhorn_eps, pre + t * n,
                          post + t * n, comb + t * n * n);
    return 0;
}

/* ------------------------------------------------------- delayed pre --- */

typedef struct {
    const uint16_t *x;        /* [T, n, C] bf16 bits                    */
    const float *pre_in;      /* [T, n]  incoming (delayed) pre-mix     */
    const float *fn;          /* [2n+n^2, n*C] projection weight        */
    const float *bias;        /* [2n+n^2]                               */
    const float *alpha;       /* [3] = pre, post, comb scales           */
    const uint16_t *norm_w;   /* [C] bf16 bits, or NULL: no fold        */
    int n, C, iters;
    double rms_eps, norm_eps, sinkhorn_eps;
    double *logits, *pre, *post, *comb; /* [T,M], [T,n], [T,n], [T,n,n] */
    float *h32;               /* [T, C] or NULL                          */
    uint16_t *layer_input;    /* [T, C] bf16 bits                        */
} pre_args;

/* One token of the delayed pre block.
 * 1. r = 1/sqrt(mean_k x_flat[k]^2 + rms_eps), x_flat[i*C + c] = x[i][c]
 *    (the sums of squares come with the projection, [A] "Approach").
 * 2. l[m] = r * (sum_k x_flat[k] fn[m][k]) * alpha_seg(m) + bias[m], with
 *    alpha_seg = alpha[0] for m < n, alpha[1] for m < 2n, alpha[2] after.
 * 3. gates and comb as in gates_from_logits.
 * 4. collapse with the INCOMING pre-mix p: h[c] = (((p0 x0 + p1 x1) + p2 x2)
 *    + p3 x3) in fp32, each product rounded.
 * 5. no fold: layer_input = bf16(h); fold: ms = mean_c h^2 (from the fp32 h),
 *    layer_input = bf16(h * 1/sqrt(ms + norm_eps) * w), one rounding. */
static void pre_token(const pre_args *a, int64_t t)
{
    const int n = a->n, C = a->C, K = n * C, M = 2 * n + n * n;
    const uint16_t *x = a->x + t * (int64_t)K;
    const float *p = a->pre_in + t * n;

    double ss = 0.0;
    for (int k = 0; k < K; ++k) {
        double v = bf16_value(x[k]);
        ss += v * v;
    }
    double r = 1.0 / sqrt(ss / (double)K + a->rms_eps);

    double *l = a->logits + t * M;
    for (int m = 0; m < M; ++m) {
        const float *w = a->fn + (int64_t)m * K;
        double dot = 0.0;
        for (int k = 0; k < K; ++k)
            dot += bf16_value(x[k]) * (double)w[k];
        double al = m < n ? a->alpha[0] : (m < 2 * n ? a->alpha[1] : a->alpha[2]);
        l[m] = r * dot * al + (double)a->bias[m];
    }
    gates_from_logits(l, n, a->iters, a->sinkhorn_eps, a->pre + t * n,
                      a->post + t * n, a->comb + t * n * n);

    float *h = (float *)malloc(sizeof(float) * (size_t)C);
    for (int c = 0; c < C; ++c) {
        float acc = p[0] * (float)bf16_value(x[c]);
        for (int i = 1; i < n; ++i) {
            float prod = p[i] * (float)bf16_value(x[(int64_t)i * C + c]);
            acc = acc + prod;
        }
        h[c] = acc;
    }
    uint16_t *out = a->layer_input + t * (int64_t)C;
    if (a->norm_w) {
        double ms = 0.0;
        for (int c = 0; c < C; ++c)
            ms += (double)h[c] * (double)h[c];
        ms /= (double)C;
        double s = 1.0 / sqrt(ms + a->norm_eps);
        for (int c = 0; c < C; ++c)
            out[c] = bf16_round((double)h[c] * s * bf16_value(a->norm_w[c]));
    } else {
        for (int c = 0; c < C; ++c)
            out[c] = bf16_round((double)h[c]);
    }
    if (a->h32)
        memcpy(a->h32 + t * (int64_t)C, h, sizeof(float) * (size_t)C);
    free(h);
}

typedef struct {
    const pre_args *args;
    int64_t t0, t1;
} pre_chunk;

static void *pre_worker(void *p)
{
    const pre_chunk *ch = (const pre_chunk *)p;
    for (int64_t t = ch->t0; t < ch->t1; ++t)
        pre_token(ch->args, t);
    return NULL;
}

/* Returns 0 on success, 1 on a bad argument.  nthreads <= 1 runs on the
 * calling thread; otherwise tokens are split into contiguous chunks, one
 * POSIX thread each (tokens are independent). */
ORACLE_API int mhc_oracle_pre_delayed(
    const uint16_t *x, const float *pre_in, const float *fn, const float *bias,
    const float *alpha, const uint16_t *norm_weight, int64_t T, int n, int C,
    int iters, double rms_eps, double norm_eps, double sinkhorn_eps,
    double *logits, double *pre, double *post, double *comb, float *h32,
    uint16_t *layer_input, int nthreads)
{
    if (T < 0 || n < 1 || C < 1 || iters < 1)
        return 1;
    if (T > 0 && (!x || !pre_in || !fn || !bias || !alpha || !logits || !pre ||
                  !post || !comb || !layer_input))
        return 1;
    pre_args a = {x, pre_in, fn, bias, alpha, norm_weight, n, C, iters,
                  rms_eps, norm_eps, sinkhorn_eps, logits, pre, post, comb,
                  h32, layer_input};
    if (nthreads <= 1 || T < 2) {
        for (int64_t t = 0; t < T; ++t)
            pre_token(&a, t);
        return 0;
    }
    if (nthreads > T)
        nthreads = (int)T;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    pre_chunk *ch = (pre_chunk *)malloc(sizeof(pre_chunk) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        ch[i].args = &a;
        ch[i].t0 = T * i / nthreads;
        ch[i].t1 = T * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, pre_worker, &ch[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(th);
    free(ch);
    return 0;
}

/* --------------------------------------------------------------- post --- */

typedef struct {
    const uint16_t *x, *y;
    const float *comb, *post;
    int n, C;
    uint16_t *x_new;
    double *x_new64;
    int64_t t0, t1;
} post_chunk;

/* x_new[t][j][c] = bf16( sum_i comb[t][i][j] * x[t][i][c] + post[t][j] * y[t][c] ),
 * evaluated exactly in fp64 from the given fp32 comb/post and bf16 x, y, then
 * rounded once ("mix the residual streams through comb and add the
 * post-gated sublayer output"; MHCPostOp in the pages). */
static void *post_worker(void *p)
{
    const post_chunk *a = (const post_chunk *)p;
    const int n = a->n, C = a->C;
    for (int64_t t = a->t0; t < a->t1; ++t) {
        const uint16_t *xt = a->x + t * (int64_t)n * C;
        const uint16_t *yt = a->y + t * (int64_t)C;
        const float *cb = a->comb + t * n * n;
        const float *pt = a->post + t * n;
        for (int j = 0; j < n; ++j) {
            for (int c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int i = 0; i < n; ++i)
                    acc += (double)cb[i * n + j] * bf16_value(xt[(int64_t)i * C + c]);
                acc += (double)pt[j] * bf16_value(yt[c]);
                int64_t o = (t * n + j) * (int64_t)C + c;
                a->x_new[o] = bf16_round(acc);
                if (a->x_new64)
                    a->x_new64[o] = acc;
            }
        }
    }
    return NULL;
}

ORACLE_API int mhc_oracle_post(const uint16_t *x, const uint16_t *y, const float *comb,
                               const float *post, int64_t T, int n, int C,
                               uint16_t *x_new, double *x_new64, int nthreads)
{
    if (T < 0 || n < 1 || C < 1)
        return 1;
    if (T > 0 && (!x || !y || !comb || !post || !x_new))
        return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > T)
        nthreads = T > 0 ? (int)T : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    post_chunk *ch = (post_chunk *)malloc(sizeof(post_chunk) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        post_chunk c = {x, y, comb, post, n, C, x_new, x_new64,
                        T * i / nthreads, T * (i + 1) / nthreads};
        ch[i] = c;
        if (nthreads == 1)
            post_worker(&ch[i]);
        else
            pthread_create(&th[i], NULL, post_worker, &ch[i]);
    }
    if (nthreads > 1)
        for (int i = 0; i < nthreads; ++i)
            pthread_join(th[i], NULL);
    free(th);
    free(ch);
    return 0;
}
