/*
 * CPU oracle for the routed-expert forward of a Kimi K2 MoE block.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU library computes.  Only the test-suite, the
 * package smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * Every floating-point value is carried in fp64 (C double).  Inputs are read
 * from the exact bytes the GPU path reads: bf16 activations as raw 16-bit
 * patterns, FP8 e4m3 weight codes as bytes, fp32 block scales and fp32 router
 * weights.
 *
 * Sources (Kimi K2 model pages, pinned revision of modeling_deepseek.py and
 * config.json):
 *   - "Input features" page, FP8 quantisation config: weights are e4m3 with
 *     one scale per 128 x 128 block; dequantised weight = code value x scale.
 *   - "SwiGLU output" page, SwiGLU MLP class: expert(x) = down(silu(gate x) * up x),
 *     three bias-free linears; gate/up map d -> d_ff, down maps d_ff -> d.
 *   - "Element-wise product" page: h = a (.) u with a = silu(gate x).
 *   - "Mixture of experts" page, moe_infer: count tokens per expert, sort the
 *     flattened (token, slot) positions by expert, run each expert on its
 *     contiguous slice, scatter the outputs back to their positions, then
 *     sum each token's k outputs weighted by topk_weight.  The page's prose:
 *     each token's output is the router-weighted sum of its selected experts
 *     plus the shared expert applied to every token.
 *   - "Input features" page, RMSNorm excerpt: the row is promoted to float32,
 *     variance = mean(h^2), h * rsqrt(variance + eps), the result is cast back
 *     to the input dtype (bf16) and multiplied by the bf16 gain (a bf16
 *     product); decoder block: hidden = residual + mlp(post_attention_norm(residual)).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - sort order of equal expert ids: ascending flat index t*k + j (stable);
 *   - counting: a histogram that adds (a token naming one expert twice is
 *     counted twice);
 *   - the activation is SiLU, silu(a) = a / (1 + exp(-a));
 *   - RMSNorm follows the excerpt's own precision: float32 arithmetic and the
 *     two bf16 roundings it writes; the variance is the exact mean of squares
 *     rounded once to float32 (a float32 sum in some order differs from it
 *     only in the last bits);
 *   - everything after RMSNorm has no intermediate rounding (the exact
 *     function; the roundings an implementation does are covered by the
 *     parity tolerance);
 *   - summation order: ((sum over j ascending of w_j * E_j(x)) + shared(x)) + residual;
 *   - dynamic FP8 activations (optional, the config's activation_scheme
 *     "dynamic" with fmt e4m3): every row entering a linear (x or the
 *     normalised row before gate/up, h before down) is quantised on the fly
 *     per group of 128 consecutive features, the K extent of a weight block:
 *     scale s = amax / 448 in float32 (1 when the group is all zero), code =
 *     the e4m3 value nearest to v / s computed in float32 (ties to the even
 *     code, magnitudes past 448 saturate), and the linear sees code * s.  h
 *     is rounded to float32 before it is quantised, the precision the
 *     decision is taken in.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits.  Exponent field 0 is subnormal: (m / 8) * 2^-6.  Otherwise
 * (1 + m / 8) * 2^(e - 7).  S.1111.111 is NaN; there are no infinities, so
 * S.1111.110 = 448 is the largest finite magnitude. */
double oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
double oracle_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double g_e4m3[256];
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

static void init_tables(void)
{
    for (int c = 0; c < 256; ++c)
        g_e4m3[c] = oracle_e4m3_value((uint8_t)c);
}

/* One quantised weight matrix [rows, cols] of e4m3 codes with fp32 scales
 * [rows/128, cols/128].  Element (r, c) dequantises to code(r, c) * scale(r/128, c/128). */
typedef struct {
    const uint8_t *q;
    const float *s;
    int64_t rows, cols;
} qmat;

static inline double wq(const qmat *m, int64_t r, int64_t c)
{
    return g_e4m3[m->q[r * m->cols + c]] * (double)m->s[(r / 128) * (m->cols / 128) + c / 128];
}

/* Dequantised element, exported so tests can compare it with a library routine. */
double oracle_dequant(const uint8_t *q, const float *s, int64_t rows, int64_t cols, int64_t r, int64_t c)
{
    pthread_once(&g_once, init_tables);
    qmat m = {q, s, rows, cols};
    return wq(&m, r, c);
}

double oracle_silu(double a)
{
    return a / (1.0 + exp(-a));
}

/* ------------------------------------------------------------------------- */
/* Dynamic FP8 activations                                                   */
/* ------------------------------------------------------------------------- */

/* The e4m3 code nearest to v: every finite non-negative code 0x00..0x7E is
 * tried, a tie goes to the code with an even mantissa, and magnitudes past
 * 448 land on 448 (the nearest finite value).  NaN gives 0x7F. */
uint8_t oracle_e4m3_encode(float v)
{
    pthread_once(&g_once, init_tables);
    if (v != v)
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    int best = 0;
    double best_dist = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double dist = fabs(g_e4m3[c] - a);
        if (dist < best_dist || (dist == best_dist && (c & 1) == 0)) {
            best = c;
            best_dist = dist;
        }
    }
    return (uint8_t)(sign | best);
}

/* One row of n features (n a multiple of 128) under the dynamic scheme:
 * out[i] = code_i * s_g for the group g = i / 128 holding i.  codes[n] and
 * scales[n / 128] receive the codes and the group scales when not NULL. */
void oracle_fp8_dynamic(int64_t n, const double *v, double *out, uint8_t *codes, float *scales)
{
    pthread_once(&g_once, init_tables);
    for (int64_t g = 0; g < n / 128; ++g) {
        const double *vg = v + g * 128;
        float amax = 0.0f;
        for (int64_t i = 0; i < 128; ++i) {
            float m = fabsf((float)vg[i]);
            if (m > amax)
                amax = m;
        }
        float s = amax / 448.0f;
        if (!(s > 0.0f))
            s = 1.0f;
        for (int64_t i = 0; i < 128; ++i) {
            float q = (float)vg[i] / s;
            uint8_t code = oracle_e4m3_encode(q);
            out[g * 128 + i] = g_e4m3[code] * (double)s;
            if (codes)
                codes[g * 128 + i] = code;
        }
        if (scales)
            scales[g] = s;
    }
}

/* ------------------------------------------------------------------------- */
/* One SwiGLU expert on one input row                                        */
/* ------------------------------------------------------------------------- */

typedef struct {
    qmat gate, up, down;   /* gate/up: [d_ff, d], down: [d, d_ff] */
} expert_t;

/* out[d] = down( silu(gate x) * (up x) ); scratch holds 3 * d_ff doubles.
 * With fp8_act the row h is quantised under the dynamic scheme before down
 * (x is the caller's, quantised already when the scheme is on). */
static void expert_row(const expert_t *ex, int64_t d, int64_t dff, const double *x, double *out, double *scratch,
                       int fp8_act)
{
    double *g = scratch, *u = scratch + dff, *h = scratch + 2 * dff;
    for (int64_t f = 0; f < dff; ++f) {
        double a = 0.0, b = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            a += wq(&ex->gate, f, c) * x[c];
            b += wq(&ex->up, f, c) * x[c];
        }
        g[f] = a;
        u[f] = b;
    }
    for (int64_t f = 0; f < dff; ++f)
        h[f] = oracle_silu(g[f]) * u[f];
    if (fp8_act) {
        oracle_fp8_dynamic(dff, h, g, NULL, NULL);
        h = g;
    }
    for (int64_t r = 0; r < d; ++r) {
        double acc = 0.0;
        for (int64_t f = 0; f < dff; ++f)
            acc += wq(&ex->down, r, f) * h[f];
        out[r] = acc;
    }
}

static expert_t make_expert(const uint8_t *const *wg, const float *const *sg, const uint8_t *const *wu,
                            const float *const *su, const uint8_t *const *wd, const float *const *sd,
                            int64_t e, int64_t d, int64_t dff)
{
    expert_t ex;
    ex.gate = (qmat){wg[e], sg[e], dff, d};
    ex.up = (qmat){wu[e], su[e], dff, d};
    ex.down = (qmat){wd[e], sd[e], d, dff};
    return ex;
}

/* Single expert on a batch of rows, for pins against a library matmul.  With
 * fp8_act each row is quantised under the dynamic scheme first. */
void oracle_expert_forward(int64_t n_rows, int64_t d, int64_t dff, const double *x, const uint8_t *wg,
                           const float *sg, const uint8_t *wu, const float *su, const uint8_t *wd,
                           const float *sd, double *out, int fp8_act)
{
    pthread_once(&g_once, init_tables);
    expert_t ex = {{wg, sg, dff, d}, {wu, su, dff, d}, {wd, sd, d, dff}};
    double *scratch = (double *)malloc(sizeof(double) * 3 * dff);
    double *xq = (double *)malloc(sizeof(double) * d);
    for (int64_t i = 0; i < n_rows; ++i) {
        const double *xi = x + i * d;
        if (fp8_act) {
            oracle_fp8_dynamic(d, xi, xq, NULL, NULL);
            xi = xq;
        }
        expert_row(&ex, d, dff, xi, out + i * d, scratch, fp8_act);
    }
    free(xq);
    free(scratch);
}

/* ------------------------------------------------------------------------- */
/* RMSNorm                                                                   */
/* ------------------------------------------------------------------------- */

/* Nearest bfloat16 to a finite binary32 value, ties to even: the upper half of
 * the pattern after adding just under half of the dropped part, plus one more
 * when the kept part is odd. */
static float bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* xn = bf16(gain * bf16(h * rsqrt(mean(h^2) + eps))), float32 arithmetic, one row. */
static void rmsnorm_row(int64_t d, const uint16_t *h_bf16, const uint16_t *gain_bf16, double eps, double *xn)
{
    double ss = 0.0;
    for (int64_t c = 0; c < d; ++c) {
        double v = oracle_bf16_value(h_bf16[c]);
        ss += v * v;
    }
    float variance = (float)(ss / (double)d);
    float inv = 1.0f / sqrtf(variance + (float)eps);
    for (int64_t c = 0; c < d; ++c) {
        float normed = bf16_round((float)oracle_bf16_value(h_bf16[c]) * inv);
        xn[c] = (double)bf16_round((float)oracle_bf16_value(gain_bf16[c]) * normed);
    }
}

void oracle_rmsnorm(int64_t n, int64_t d, const uint16_t *h_bf16, const uint16_t *gain_bf16, double eps, double *xn)
{
    for (int64_t t = 0; t < n; ++t)
        rmsnorm_row(d, h_bf16 + t * d, gain_bf16, eps, xn + t * d);
}

/* ------------------------------------------------------------------------- */
/* Routing plan: histogram, exclusive scan, stable order by expert           */
/* ------------------------------------------------------------------------- */

/* counts[E], offsets[E+1], sorted_pos[n*k], inv_pos[n*k].
 * sorted_pos[i] = flat index (t*k + j) of the i-th entry when entries are
 * ordered by (expert id, flat index).  inv_pos[p] = i with sorted_pos[i] = p.
 * Entries whose id lies outside [0, E) are left out: inv_pos = -1 and the tail
 * of sorted_pos beyond offsets[E] is -1.  Returns the number of such entries. */
int64_t oracle_permute(int64_t n, int64_t k, int64_t E, const int32_t *ids, int32_t *counts, int32_t *offsets,
                       int32_t *sorted_pos, int32_t *inv_pos)
{
    int64_t R = n * k, bad = 0;
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t p = 0; p < R; ++p) {
        if (ids[p] >= 0 && ids[p] < E)
            counts[ids[p]] += 1;
        else
            bad += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int64_t e = 0; e < E; ++e)
        next[e] = offsets[e];
    for (int64_t p = 0; p < R; ++p) {
        int32_t e = ids[p];
        if (e >= 0 && e < E) {
            sorted_pos[next[e]] = (int32_t)p;
            inv_pos[p] = next[e];
            next[e] += 1;
        } else {
            inv_pos[p] = -1;
        }
    }
    for (int64_t i = offsets[E]; i < R; ++i)
        sorted_pos[i] = -1;
    free(next);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Routed forward, token by token (brute force)                              */
/* ------------------------------------------------------------------------- */

typedef struct {
    int64_t d, dff, k, E;
    const uint16_t *x;            /* [N, d] bf16: expert input rows */
    const int32_t *ids;           /* [N, k] */
    const float *w;               /* [N, k] */
    const uint8_t *const *wg, *const *wu, *const *wd;   /* per-expert pointers (NULL if unused) */
    const float *const *sg, *const *su, *const *sd;
    /* full block only */
    const uint16_t *resid;        /* [N, d] bf16 residual, or NULL */
    const uint16_t *gain;         /* [d] bf16: x is the residual, normalised first */
    double eps;
    const uint8_t *shg, *shu, *shd;  /* shared expert, or NULL */
    const float *ssg, *ssu, *ssd;
    int64_t dff_sh;
    int fp8_act;                  /* dynamic FP8 activations */
    /* work */
    const int64_t *tok;           /* token indices to evaluate */
    int64_t n_tok;
    double *y;                    /* [n_tok, d] */
    int64_t next;                 /* shared work counter */
    pthread_mutex_t mu;
} job_t;

static int64_t take(job_t *jb)
{
    pthread_mutex_lock(&jb->mu);
    int64_t i = jb->next++;
    pthread_mutex_unlock(&jb->mu);
    return i;
}

static void *token_worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    int64_t d = jb->d, dff = jb->dff, k = jb->k;
    int64_t smax = dff > jb->dff_sh ? dff : jb->dff_sh;
    double *xin = (double *)malloc(sizeof(double) * d);
    double *o = (double *)malloc(sizeof(double) * d);
    double *scratch = (double *)malloc(sizeof(double) * 3 * (smax > 0 ? smax : 1));
    for (;;) {
        int64_t i = take(jb);
        if (i >= jb->n_tok)
            break;
        int64_t t = jb->tok[i];
        double *acc = jb->y + i * d;
        if (jb->gain)
            rmsnorm_row(d, jb->x + t * d, jb->gain, jb->eps, xin);
        else
            for (int64_t c = 0; c < d; ++c)
                xin[c] = oracle_bf16_value(jb->x[t * d + c]);
        if (jb->fp8_act)
            oracle_fp8_dynamic(d, xin, xin, NULL, NULL);
        for (int64_t c = 0; c < d; ++c)
            acc[c] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            int32_t e = jb->ids[t * k + j];
            if (e < 0 || e >= jb->E)
                continue;
            expert_t ex = make_expert(jb->wg, jb->sg, jb->wu, jb->su, jb->wd, jb->sd, e, d, dff);
            expert_row(&ex, d, dff, xin, o, scratch, jb->fp8_act);
            double wt = (double)jb->w[t * k + j];
            for (int64_t c = 0; c < d; ++c)
                acc[c] += wt * o[c];
        }
        if (jb->shg) {
            expert_t sh = {{jb->shg, jb->ssg, jb->dff_sh, d}, {jb->shu, jb->ssu, jb->dff_sh, d},
                           {jb->shd, jb->ssd, d, jb->dff_sh}};
            expert_row(&sh, d, jb->dff_sh, xin, o, scratch, jb->fp8_act);
            for (int64_t c = 0; c < d; ++c)
                acc[c] += o[c];
        }
        if (jb->resid)
            for (int64_t c = 0; c < d; ++c)
                acc[c] += oracle_bf16_value(jb->resid[t * d + c]);
    }
    free(xin);
    free(o);
    free(scratch);
    return NULL;
}

static void run_job(job_t *jb, int nthreads)
{
    pthread_once(&g_once, init_tables);
    if (nthreads < 1)
        nthreads = 1;
    jb->next = 0;
    pthread_mutex_init(&jb->mu, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i)
        pthread_create(&th[i], NULL, token_worker, jb);
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&jb->mu);
}

/* y[i, :] = sum_j topk_weight[t, j] * expert_{ids[t, j]}(x[t, :]) for t = tok[i].
 * Expert pointer tables are indexed by expert id; entries of experts that
 * no selected token uses may be NULL. */
void oracle_moe_infer(int64_t d, int64_t dff, int64_t k, int64_t E, const uint16_t *x, const int32_t *ids,
                      const float *w, const uint8_t *const *wg, const float *const *sg, const uint8_t *const *wu,
                      const float *const *su, const uint8_t *const *wd, const float *const *sd,
                      const int64_t *tok, int64_t n_tok, double *y, int nthreads, int fp8_act)
{
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.d = d; jb.dff = dff; jb.k = k; jb.E = E; jb.fp8_act = fp8_act;
    jb.x = x; jb.ids = ids; jb.w = w;
    jb.wg = wg; jb.sg = sg; jb.wu = wu; jb.su = su; jb.wd = wd; jb.sd = sd;
    jb.tok = tok; jb.n_tok = n_tok; jb.y = y;
    run_job(&jb, nthreads);
}

/* Full block for the selected tokens:
 * y = h + ( sum_j w_j * E_j(xn) + S(xn) ),  xn = RMSNorm(h) with gain and eps.
 * The shared expert pointers may be NULL (no shared expert). */
void oracle_layer_forward(int64_t d, int64_t dff, int64_t k, int64_t E, const uint16_t *hidden,
                          const uint16_t *gain, double eps, const int32_t *ids, const float *w,
                          const uint8_t *const *wg, const float *const *sg, const uint8_t *const *wu,
                          const float *const *su, const uint8_t *const *wd, const float *const *sd,
                          const uint8_t *shg, const float *ssg, const uint8_t *shu, const float *ssu,
                          const uint8_t *shd, const float *ssd, int64_t dff_sh, const int64_t *tok,
                          int64_t n_tok, double *y, int nthreads, int fp8_act)
{
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.d = d; jb.dff = dff; jb.k = k; jb.E = E; jb.fp8_act = fp8_act;
    jb.x = hidden; jb.ids = ids; jb.w = w;
    jb.wg = wg; jb.sg = sg; jb.wu = wu; jb.su = su; jb.wd = wd; jb.sd = sd;
    jb.resid = hidden; jb.gain = gain; jb.eps = eps;
    jb.shg = shg; jb.shu = shu; jb.shd = shd; jb.ssg = ssg; jb.ssu = ssu; jb.ssd = ssd;
    jb.dff_sh = shg ? dff_sh : 0;
    jb.tok = tok; jb.n_tok = n_tok; jb.y = y;
    run_job(&jb, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Routed forward the way the "Mixture of experts" page's moe_infer does it  */
/* ------------------------------------------------------------------------- */

/* Sorted-slice form: count, sort the flat positions by expert, gather the
 * token rows into that order, run each expert on its contiguous slice, write
 * each output row back to its flat position, then sum each token's k rows
 * weighted by topk_weight.  Used on small inputs to pin oracle_moe_infer:
 * the per-row arithmetic and the summation order are the same, so the two
 * must agree bit for bit.  y is [n, d]. */
void oracle_moe_infer_sorted(int64_t n, int64_t d, int64_t dff, int64_t k, int64_t E, const uint16_t *x,
                             const int32_t *ids, const float *w, const uint8_t *const *wg,
                             const float *const *sg, const uint8_t *const *wu, const float *const *su,
                             const uint8_t *const *wd, const float *const *sd, double *y, int fp8_act)
{
    pthread_once(&g_once, init_tables);
    int64_t R = n * k;
    int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t *idxs = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    oracle_permute(n, k, E, ids, counts, offsets, idxs, inv);
    double *sorted_tokens = (double *)malloc(sizeof(double) * (size_t)(R * d));
    double *outs = (double *)malloc(sizeof(double) * (size_t)(R * d));
    double *new_x = (double *)calloc((size_t)(R * d), sizeof(double));
    double *scratch = (double *)malloc(sizeof(double) * 3 * dff);
    int64_t nvalid = offsets[E];
    for (int64_t i = 0; i < nvalid; ++i) {
        int64_t t = idxs[i] / k;
        for (int64_t c = 0; c < d; ++c)
            sorted_tokens[i * d + c] = oracle_bf16_value(x[t * d + c]);
        if (fp8_act)
            oracle_fp8_dynamic(d, sorted_tokens + i * d, sorted_tokens + i * d, NULL, NULL);
    }
    int64_t start = 0;
    for (int64_t e = 0; e < E; ++e) {
        int64_t end = start + counts[e];
        if (counts[e] == 0)
            continue;
        expert_t ex = make_expert(wg, sg, wu, su, wd, sd, e, d, dff);
        for (int64_t i = start; i < end; ++i)
            expert_row(&ex, d, dff, sorted_tokens + i * d, outs + i * d, scratch, fp8_act);
        start = end;
    }
    for (int64_t i = 0; i < nvalid; ++i)
        memcpy(new_x + (int64_t)idxs[i] * d, outs + i * d, sizeof(double) * (size_t)d);
    for (int64_t t = 0; t < n; ++t) {
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; ++j)
                acc += (double)w[t * k + j] * new_x[(t * k + j) * d + c];
            y[t * d + c] = acc;
        }
    }
    free(counts); free(offsets); free(idxs); free(inv);
    free(sorted_tokens); free(outs); free(new_x); free(scratch);
}
