/*
 * coat_oracle.c -- plain float64 CPU reference for the fused FP8 AdamW step
 * with Dynamic Range Expansion (DRE).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, table or constant
 * generator with the CUDA library.
 *
 * Sources (all on the COAT paper-review page, "COAT: Compressing Optimizer
 * States and Activation for Memory-Efficient FP8 Training", xllm-io blog):
 *   - FP8 quantization:   section 3 (技术架构), core formulas, "FP8量化":
 *       X_FP8 = round(X_FP32 / S_X),  S_X = max|X_FP32| / Delta_max^E4M3
 *   - AdamW update rule:  section 3, core formulas, "AdamW优化器更新规则":
 *       m_t = b1 m_{t-1} + (1-b1) g,  v_t = b2 v_{t-1} + (1-b2) g^2,
 *       mhat = m_t/(1-b1^t), vhat = v_t/(1-b2^t),
 *       w_{t+1} = w_t - lr (mhat/(sqrt(vhat)+eps) + wd w_t)
 *   - Dynamic Range Expansion: section 3, "动态范围扩展":
 *       f(x) = sign(x)|x|^k,  R_f(X) = (max|X|/min|X|)^k = R_X^k,
 *       optimal k solves R_X^k = R_E4M3, i.e. k = log_{R_X}(R_E4M3)
 *   - the optimizer states are the quantized tensors (section 4 table, DRE
 *     row: DRE reshapes the optimizer-state distribution to fit FP8), one
 *     (S, k) pair per group of G contiguous elements.
 *
 * Readings where the page is silent (each one is listed in the design notes):
 *   - E4M3 is the OCP "E4M3FN" format: bias 7, no infinities, 0x7F/0xFF NaN,
 *     Delta_max = 448, smallest subnormal 2^-9.
 *   - R_E4M3 is a parameter; the library's value is 448 / 2^-9 = 229376.
 *   - min|X| is taken over the non-zero elements of the group.
 *   - all-zero group: k = 1, S = 0, every code 0x00.
 *   - R_X = 1 (one non-zero magnitude): k = 1.
 *   - k = min(log(R_E4M3)/log(R_X), K_CAP) with K_CAP = 8, then capped so
 *     that S = max^k / 448 stays inside [2^-125, 2^126] (normal fp32).
 *   - k and S are stored as fp32; S and the codes are computed from the
 *     stored (fp32-rounded) k.
 *   - round(.) is round-to-nearest, ties to the even code, saturating at
 *     +-448; zero always encodes as 0x00.
 *   - the gradient of the current step is used (the page's g_{t-1} index is
 *     read as "the gradient passed with this step").
 *   - weight decay is decoupled and uses w_t before the update.
 *   - the update uses the fp32 m_t, v_t; quantization is for storage.
 *   - the dequantized states, the new states and the new weights are fp32
 *     values (the page calls the dequantized tensor X_FP32).
 *   - hyper-parameters arrive as fp32 and are used at that exact value.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_DELTA_MAX 448.0
#define ORACLE_K_CAP 8.0
#define ORACLE_S_LOG2_MIN (-125.0)
#define ORACLE_S_LOG2_MAX (126.0)

/* ------------------------------------------------------------------ */
/* E4M3 codec from the bit definition                                  */
/* ------------------------------------------------------------------ */

/* Value of an 8-bit E4M3 code: sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits.  Exponent field 0 is subnormal: (mant/8) * 2^-6.  The two
 * codes with all exponent and mantissa bits set are NaN. */
double coat_oracle_e4m3_decode(int code)
{
    int c = code & 0xFF;
    int sign = c >> 7;
    int expo = (c >> 3) & 0xF;
    int mant = c & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

static double g_pos_values[127]; /* values of codes 0x00 .. 0x7E */
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;

static void build_pos_values(void)
{
    for (int c = 0; c < 127; ++c)
        g_pos_values[c] = coat_oracle_e4m3_decode(c);
}

/* Nearest E4M3 code to y: scan every finite non-negative code for the one
 * closest to |y|; on an exact tie keep the code with the even mantissa.
 * Values beyond 448 have 448 as their nearest finite code, which is the
 * saturating behaviour.  A magnitude that rounds to zero gives 0x00 whatever
 * its sign. */
int coat_oracle_e4m3_encode(double y)
{
    pthread_once(&g_table_once, build_pos_values);
    double a = fabs(y);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 127; ++c) {
        double d = fabs(a - g_pos_values[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best_d = d;
            best = c;
        }
    }
    if (best == 0)
        return 0;
    return (y < 0.0 ? 0x80 : 0x00) | best;
}

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* DRE on one group                                                    */
/* ------------------------------------------------------------------ */

typedef struct {
    double k_formula; /* log(R_E4M3)/log(R_X) before any cap (inf if R_X==1, 0 if empty) */
    double k_exact;   /* after the cap and the S-range guard, before fp32 rounding */
    float k32;        /* stored exponent */
    float S32;        /* stored scale */
    double maxabs;
    double minabs;    /* smallest non-zero magnitude (0 if none) */
} dre_params;

/* k and S for a group of fp32 values (section 3, Dynamic Range Expansion:
 * R_X = max|X|/min|X|, k = log_{R_X}(R_E4M3), S = max|f(X)|/448 with
 * f(x) = sign(x)|x|^k, so max|f(X)| = max|X|^k). */
static dre_params dre_group_params(const float *x, int64_t n, double R)
{
    dre_params p;
    double mx = 0.0, mn = INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        double a = fabs((double)x[i]);
        if (a > mx)
            mx = a;
        if (a != 0.0 && a < mn)
            mn = a;
    }
    p.maxabs = mx;
    if (mx == 0.0) {
        p.minabs = 0.0;
        p.k_formula = 0.0;
        p.k_exact = 1.0;
        p.k32 = 1.0f;
        p.S32 = 0.0f;
        return p;
    }
    p.minabs = mn;
    double k;
    if (mn == mx) {
        p.k_formula = INFINITY;
        k = 1.0;
    } else {
        p.k_formula = log(R) / log(mx / mn);
        k = p.k_formula < ORACLE_K_CAP ? p.k_formula : ORACLE_K_CAP;
    }
    /* keep S = mx^k / 448 a normal fp32 number */
    double l = log2(mx);
    double l448 = log2(ORACLE_DELTA_MAX);
    if (l < 0.0) {
        double bound = (l448 + ORACLE_S_LOG2_MIN) / l;
        if (bound < k)
            k = bound;
    } else if (l > 0.0) {
        double bound = (l448 + ORACLE_S_LOG2_MAX) / l;
        if (bound < k)
            k = bound;
    }
    p.k_exact = k;
    p.k32 = (float)k;
    p.S32 = (float)(pow(mx, (double)p.k32) / ORACLE_DELTA_MAX);
    return p;
}

/* Expanded and scaled value f(x)/S = 448 sign(x) (|x|/max)^k, in float64. */
static double dre_scaled(double x, const dre_params *p)
{
    if (x == 0.0 || p->maxabs == 0.0)
        return 0.0;
    double r = pow(fabs(x) / p->maxabs, (double)p->k32) * ORACLE_DELTA_MAX;
    return x < 0.0 ? -r : r;
}

/* Inverse of the quantizer: f^{-1}(dec(q) * S) = sign(q)(|dec(q)| S)^(1/k),
 * rounded to fp32 (the page's X_FP32). */
static float dre_dequant_one(int code, float S, float k)
{
    double d = coat_oracle_e4m3_decode(code);
    double a = fabs(d) * (double)S;
    if (a == 0.0)
        return d < 0.0 ? -0.0f : 0.0f;
    double r = pow(a, 1.0 / (double)k);
    return (float)(d < 0.0 ? -r : r);
}

/* One group in full detail (for the self-tests). */
int coat_oracle_dre_group(const float *x, int64_t n, double R, double *k_formula,
                          double *k_exact, float *k32, float *S32, double *y, uint8_t *q)
{
    if (n <= 0 || !(R > 1.0))
        return 1;
    dre_params p = dre_group_params(x, n, R);
    if (k_formula) *k_formula = p.k_formula;
    if (k_exact) *k_exact = p.k_exact;
    if (k32) *k32 = p.k32;
    if (S32) *S32 = p.S32;
    for (int64_t i = 0; i < n; ++i) {
        double yi = dre_scaled((double)x[i], &p);
        if (y) y[i] = yi;
        if (q) q[i] = (uint8_t)coat_oracle_e4m3_encode(yi);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* threading over groups                                               */
/* ------------------------------------------------------------------ */

typedef void (*group_fn)(void *ctx, int64_t g0, int64_t g1);

typedef struct {
    group_fn fn;
    void *ctx;
    int64_t g0, g1;
} worker_arg;

static void *worker_main(void *a)
{
    worker_arg *w = (worker_arg *)a;
    w->fn(w->ctx, w->g0, w->g1);
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0)
        return nthreads;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

static void run_groups(group_fn fn, void *ctx, int64_t ngroups, int nthreads)
{
    int t = resolve_threads(nthreads);
    if ((int64_t)t > ngroups)
        t = (int)(ngroups > 0 ? ngroups : 1);
    if (t <= 1) {
        fn(ctx, 0, ngroups);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)t);
    worker_arg *args = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)t);
    int64_t per = (ngroups + t - 1) / t;
    int started = 0;
    for (int i = 0; i < t; ++i) {
        int64_t a = (int64_t)i * per, b = a + per;
        if (a >= ngroups)
            break;
        if (b > ngroups)
            b = ngroups;
        args[i].fn = fn;
        args[i].ctx = ctx;
        args[i].g0 = a;
        args[i].g1 = b;
        if (pthread_create(&th[i], NULL, worker_main, &args[i]) != 0) {
            fn(ctx, a, b); /* run inline if a thread cannot start */
            args[i].fn = NULL;
        }
        started = i + 1;
    }
    for (int i = 0; i < started; ++i)
        if (args[i].fn)
            pthread_join(th[i], NULL);
    free(th);
    free(args);
}

/* ------------------------------------------------------------------ */
/* standalone quantize / dequantize over a flat buffer                 */
/* ------------------------------------------------------------------ */

typedef struct {
    const float *x;
    int64_t n;
    int32_t G;
    double R;
    uint8_t *q;
    float *S;
    float *k;
} quant_ctx;

static void quant_groups(void *c, int64_t g0, int64_t g1)
{
    quant_ctx *q = (quant_ctx *)c;
    for (int64_t g = g0; g < g1; ++g) {
        int64_t b = g * q->G, e = b + q->G;
        if (e > q->n)
            e = q->n;
        dre_params p = dre_group_params(q->x + b, e - b, q->R);
        q->S[g] = p.S32;
        q->k[g] = p.k32;
        for (int64_t i = b; i < e; ++i)
            q->q[i] = (uint8_t)coat_oracle_e4m3_encode(dre_scaled((double)q->x[i], &p));
    }
}

int coat_oracle_dre_quantize(const float *x, int64_t n, int32_t G, double R, uint8_t *q,
                             float *S, float *k, int nthreads)
{
    if (n <= 0 || G <= 0 || !(R > 1.0) || !x || !q || !S || !k)
        return 1;
    quant_ctx c = {x, n, G, R, q, S, k};
    run_groups(quant_groups, &c, (n + G - 1) / G, nthreads);
    return 0;
}

/* FP8 quantization without the expansion (section 3, the FP8 quantization
 * equation alone): S = max|X| / 448 rounded to float, q = E4M3(X / S). */
typedef struct {
    const float *x;
    int64_t n;
    int32_t G;
    uint8_t *q;
    float *S;
} absmax_ctx;

static void absmax_groups(void *c, int64_t g0, int64_t g1)
{
    absmax_ctx *a = (absmax_ctx *)c;
    for (int64_t g = g0; g < g1; ++g) {
        int64_t b = g * a->G, e = b + a->G;
        if (e > a->n)
            e = a->n;
        double mx = 0.0;
        for (int64_t i = b; i < e; ++i)
            if (fabs((double)a->x[i]) > mx)
                mx = fabs((double)a->x[i]);
        float S32 = (float)(mx / 448.0);
        a->S[g] = S32;
        for (int64_t i = b; i < e; ++i)
            a->q[i] = (uint8_t)(S32 > 0.0f ? coat_oracle_e4m3_encode((double)a->x[i] / (double)S32)
                                           : 0);
    }
}

int coat_oracle_absmax_quantize(const float *x, int64_t n, int32_t G, uint8_t *q, float *S,
                                int nthreads)
{
    if (n <= 0 || G <= 0 || !x || !q || !S)
        return 1;
    absmax_ctx c = {x, n, G, q, S};
    run_groups(absmax_groups, &c, (n + G - 1) / G, nthreads);
    return 0;
}

typedef struct {
    const uint8_t *q;
    const float *S;
    const float *k;
    int64_t n;
    int32_t G;
    float *x;
} dequant_ctx;

static void dequant_groups(void *c, int64_t g0, int64_t g1)
{
    dequant_ctx *d = (dequant_ctx *)c;
    for (int64_t g = g0; g < g1; ++g) {
        int64_t b = g * d->G, e = b + d->G;
        if (e > d->n)
            e = d->n;
        for (int64_t i = b; i < e; ++i)
            d->x[i] = dre_dequant_one(d->q[i], d->S[g], d->k[g]);
    }
}

int coat_oracle_dre_dequantize(const uint8_t *q, const float *S, const float *k, int64_t n,
                               int32_t G, float *x, int nthreads)
{
    if (n <= 0 || G <= 0 || !x || !q || !S || !k)
        return 1;
    dequant_ctx c = {q, S, k, n, G, x};
    run_groups(dequant_groups, &c, (n + G - 1) / G, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* the fused AdamW + DRE step                                          */
/* ------------------------------------------------------------------ */

typedef struct {
    float *w;
    const uint16_t *g;
    uint8_t *mq, *vq;
    float *meta; /* per group: S_m, k_m, S_v, k_v */
    int64_t n;
    int32_t G;
    double b1, b2, lr, eps, wd, bc1, bc2, R;
} step_ctx;

static void step_groups(void *c, int64_t g0, int64_t g1)
{
    step_ctx *s = (step_ctx *)c;
    float *mbuf = (float *)malloc(sizeof(float) * (size_t)s->G);
    float *vbuf = (float *)malloc(sizeof(float) * (size_t)s->G);
    for (int64_t g = g0; g < g1; ++g) {
        int64_t b = g * s->G, e = b + s->G;
        if (e > s->n)
            e = s->n;
        float *meta = s->meta + 4 * g;
        for (int64_t i = b; i < e; ++i) {
            /* previous states, dequantized to fp32 */
            double m_prev = dre_dequant_one(s->mq[i], meta[0], meta[1]);
            double v_prev = dre_dequant_one(s->vq[i], meta[2], meta[3]);
            double gi = bf16_to_double(s->g[i]);
            /* AdamW (section 3 core formulas) */
            float m = (float)(s->b1 * m_prev + (1.0 - s->b1) * gi);
            float v = (float)(s->b2 * v_prev + (1.0 - s->b2) * gi * gi);
            double mhat = (double)m / s->bc1;
            double vhat = (double)v / s->bc2;
            double w = (double)s->w[i];
            s->w[i] = (float)(w - s->lr * (mhat / (sqrt(vhat) + s->eps) + s->wd * w));
            mbuf[i - b] = m;
            vbuf[i - b] = v;
        }
        /* re-quantize both moments with fresh DRE parameters */
        dre_params pm = dre_group_params(mbuf, e - b, s->R);
        dre_params pv = dre_group_params(vbuf, e - b, s->R);
        for (int64_t i = b; i < e; ++i) {
            s->mq[i] = (uint8_t)coat_oracle_e4m3_encode(dre_scaled((double)mbuf[i - b], &pm));
            s->vq[i] = (uint8_t)coat_oracle_e4m3_encode(dre_scaled((double)vbuf[i - b], &pv));
        }
        meta[0] = pm.S32;
        meta[1] = pm.k32;
        meta[2] = pv.S32;
        meta[3] = pv.k32;
    }
    free(mbuf);
    free(vbuf);
}

int coat_oracle_adamw_step(float *w, const uint16_t *g, uint8_t *mq, uint8_t *vq, float *meta,
                           int64_t n, int32_t G, float beta1, float beta2, float lr, float eps,
                           float weight_decay, int64_t step, double R, int nthreads)
{
    if (n <= 0 || G <= 0 || step < 1 || !(R > 1.0) || !w || !g || !mq || !vq || !meta)
        return 1;
    step_ctx c;
    c.w = w;
    c.g = g;
    c.mq = mq;
    c.vq = vq;
    c.meta = meta;
    c.n = n;
    c.G = G;
    c.b1 = (double)beta1;
    c.b2 = (double)beta2;
    c.lr = (double)lr;
    c.eps = (double)eps;
    c.wd = (double)weight_decay;
    c.bc1 = 1.0 - pow(c.b1, (double)step);
    c.bc2 = 1.0 - pow(c.b2, (double)step);
    c.R = R;
    run_groups(step_groups, &c, (n + G - 1) / G, nthreads);
    return 0;
}

int coat_oracle_threads(int nthreads)
{
    return resolve_threads(nthreads);
}
