/*
 * Plain fp64 CPU oracle of the token-choice MoE feed-forward block
 * (AFMoE, and the MiniMax-M3 variant).
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code with the CUDA path.
 *
 * Every value is upcast exactly to double on load and all arithmetic is done
 * in double.  Tokens are independent, so the outer loop over tokens is split
 * across threads; each token's result is computed by one thread in a fixed
 * order, so results do not depend on the thread count.
 *
 * Steps, for each token x (a row of X):
 *   1. router logits l_e = sum_h x_h * Wr[e,h]
 *        ("Checkpoint weight layout", Arcee AFMoE issue: the router is
 *         mlp.router.gate; HF AFMoE docs, "expert routing": each token picks
 *         its top-k experts from the router logits)
 *   2. scores s_e = sigmoid(l_e), or softmax over e
 *        ("Routing detail", Arcee AFMoE issue: score_func sigmoid; HF AFMoE
 *         docs, key features: sigmoid or softmax routing)
 *   3. biased scores c_e = s_e + b_e, used for selection only
 *        ("Routing detail": expert_bias added for selection only;
 *         MiniMax-M3 issue, "Architecture specification": e_score_correction_bias)
 *   4. the k experts with the largest c, in descending c; equal c -> lower
 *      expert index first (the pages do not fix a tie rule: lowest index)
 *   5. weights gathered from the UNBIASED scores, w_j = s_{idx_j}; if
 *      route_norm, w_j /= sum_j w_j; then w_j *= route_scale
 *        ("Routing detail": weights from the unbiased scores, then route_norm
 *         renormalisation and a route_scale multiply)
 *   6. each selected expert e: g = Wg[e] x, u = Wu[e] x, a = act(g, u),
 *      y_e = Wd[e] a; weights are stored per expert as [out, in]
 *        ("Checkpoint weight layout": experts.{gate,up,down}_proj pre-stacked)
 *      act = silu:      a = g * sigmoid(g) * u
 *        (HF AFMoE docs, AfmoeConfig: hidden_act default "silu")
 *      act = swigluoai: g' = min(g, limit), u' = clamp(u, -limit, limit),
 *                       a = g' * sigmoid(alpha g') * (u' + beta)
 *        (MiniMax-M3 issue, "Architecture specification", Activation bullet;
 *         where the clamp applies is not printed: the gpt-oss convention it
 *         names is taken)
 *   7. shared experts, always on with weight 1.0: one MLP of total width S
 *      (separate tensors), or the packed slice at index E of the stacked
 *      tensors (MiniMax-M3 issue: packed shared expert, fixed score 1.0)
 *        (HF AFMoE docs, "shared experts"; AfmoeConfig num_shared_experts)
 *   8. Y = sum_j w_j y_{idx_j} + y_shared
 *
 * Also, for the layers around and before the block:
 *   - dense MLP of width W (the dense prefix layers: a plain MLP;
 *       Arcee AFMoE issue, "Dense prefix"; HF AFMoE docs, AfmoeConfig
 *       intermediate_size and num_dense_layers; MiniMax-M3 issue,
 *       "Architecture specification": dense_intermediate_size), the same
 *       expert MLP as step 6 with the layer's weights;
 *   - RMSNorm of a row, y_h = x_h / sqrt(mean_h x_h^2 + eps) * g_h with
 *       g = w, or g = 1 + w (Gemma style)
 *       (Arcee AFMoE issue: pre_mlp_layernorm / post_mlp_layernorm in a
 *        sandwich; HF AFMoE docs, AfmoeConfig rms_norm_eps; MiniMax-M3 issue:
 *        Gemma-style RMSNorm, weight + 1, on all norms).
 *
 * Block-scaled expert weights (the pages' checkpoints are 4-bit (Arcee AFMoE
 * issue, "Checkpoint confirmed") and MXFP8 (MiniMax-M3 issue, "Validation")):
 * an element is decoded exactly to double and multiplied by its block's scale,
 * following the OCP Microscaling Formats (MX) v1.0 specification:
 *   - E8M0 scale: 2^(s - 127); s = 255 is NaN;
 *   - E4M3 element (MXFP8): sign, 4 exponent bits (bias 7), 3 mantissa bits;
 *       exponent 0 is subnormal (2^-6 * m/8); S.1111.111 is NaN, no infinities;
 *   - E2M1 element (MXFP4): sign, 2 exponent bits (bias 1), 1 mantissa bit;
 *       exponent 0 is subnormal (m/2): the values 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 *   - one scale per 32 consecutive elements along the reduction index.
 * Storage (this library's reading; the pages give no layout): element codes
 * row-major like the bf16 tensors, one per byte (E4M3) or two per byte (E2M1,
 * element 2j in the low nibble); scales of a [rows, cols] matrix block-major,
 * scale[(c / 32) * rows + r] for element (r, c).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_MXFP8 = 2, OR_MXFP4 = 3 };
enum { OR_SIGMOID = 0, OR_SOFTMAX = 1 };
enum { OR_SILU = 0, OR_SWIGLU_OAI = 1 };

typedef struct {
    int H, E, k;
    int I;             /* routed expert width (moe_intermediate_size) */
    int S;             /* total shared width; 0 = no shared expert */
    int shared_packed; /* 1: shared expert is slice E of the stacked tensors (width I) */
    int score_func;
    int route_norm;
    double route_scale;
    int act;
    double alpha, limit, beta;
} oracle_cfg;

static double ld(const void *p, int dtype, size_t i)
{
    if (dtype == OR_BF16) {
        uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return (double)((const float *)p)[i];
}

static double e8m0(uint8_t s) { return s == 255 ? NAN : ldexp(1.0, (int)s - 127); }

static double e4m3(uint8_t b)
{
    const int e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (b & 0x80) ? -v : v;
}

static double e2m1(uint8_t n)
{
    const int e = (n >> 1) & 3, m = n & 1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return (n & 8) ? -v : v;
}

/* Element (r, c) of a [rows, cols] weight matrix (c: the reduction index) of
 * dtype wd; scale: the MX block scales (block-major), or NULL. */
static double wget(const void *q, const uint8_t *scale, int wd, size_t r, size_t c, size_t rows, size_t cols)
{
    const size_t i = r * cols + c;
    if (wd == OR_MXFP8) return e8m0(scale[(c / 32) * rows + r]) * e4m3(((const uint8_t *)q)[i]);
    if (wd == OR_MXFP4) {
        const uint8_t b = ((const uint8_t *)q)[i / 2];
        return e8m0(scale[(c / 32) * rows + r]) * e2m1((uint8_t)((i & 1) ? b >> 4 : b & 15));
    }
    return ld(q, wd, i);
}

/* bytes of n elements of dtype wd (n even for E2M1) */
static size_t wbytes(int wd, size_t n)
{
    return wd == OR_F32 ? 4 * n : wd == OR_BF16 ? 2 * n : wd == OR_MXFP8 ? n : n / 2;
}

static int mx(int wd) { return wd == OR_MXFP8 || wd == OR_MXFP4; }

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

double oracle_act(const oracle_cfg *c, double g, double u)
{
    if (c->act == OR_SWIGLU_OAI) {
        double gc = g > c->limit ? c->limit : g;
        double uc = u > c->limit ? c->limit : (u < -c->limit ? -c->limit : u);
        return gc * sigmoid(c->alpha * gc) * (uc + c->beta);
    }
    return g * sigmoid(g) * u;
}

/* Routing of one token.  x: H values of dtype xd.  Outputs (any may be NULL):
 * logits[E], scores[E], biased[E], idx[k], w[k], margin (c_(k) - c_(k+1),
 * +inf when k == E). */
static void route_token(const oracle_cfg *c, const void *X, int xd, size_t row,
                        const float *Wr, const float *bias, double *logits, double *scores,
                        double *biased, int *idx, double *w, double *margin)
{
    const int E = c->E, H = c->H, k = c->k;
    double *l = (double *)malloc(sizeof(double) * E * 3);
    double *s = l + E, *cb = s + E;
    int *order = (int *)malloc(sizeof(int) * E);

    for (int e = 0; e < E; e++) {
        double acc = 0.0;
        for (int h = 0; h < H; h++)
            acc += ld(X, xd, row * (size_t)H + h) * (double)Wr[(size_t)e * H + h];
        l[e] = acc;
    }
    if (c->score_func == OR_SOFTMAX) {
        double m = l[0], z = 0.0;
        for (int e = 1; e < E; e++) m = l[e] > m ? l[e] : m;
        for (int e = 0; e < E; e++) z += exp(l[e] - m);
        for (int e = 0; e < E; e++) s[e] = exp(l[e] - m) / z;
    } else {
        for (int e = 0; e < E; e++) s[e] = sigmoid(l[e]);
    }
    for (int e = 0; e < E; e++) cb[e] = s[e] + (bias ? (double)bias[e] : 0.0);

    /* insertion sort of expert ids: larger c first, equal c -> lower id first */
    for (int e = 0; e < E; e++) {
        int j = e;
        while (j > 0 && (cb[order[j - 1]] < cb[e])) {
            order[j] = order[j - 1];
            j--;
        }
        order[j] = e;
    }

    if (idx || w) {
        double sum = 0.0;
        for (int j = 0; j < k; j++) sum += s[order[j]];
        for (int j = 0; j < k; j++) {
            double wj = s[order[j]];
            if (c->route_norm) wj = wj / sum;
            wj = wj * c->route_scale;
            if (idx) idx[j] = order[j];
            if (w) w[j] = wj;
        }
    }
    if (margin) *margin = (k < E) ? cb[order[k - 1]] - cb[order[k]] : INFINITY;
    for (int e = 0; e < E; e++) {
        if (logits) logits[e] = l[e];
        if (scores) scores[e] = s[e];
        if (biased) biased[e] = cb[e];
    }
    free(order);
    free(l);
}

/* One expert MLP of width W on one token: g = Wg x, u = Wu x, a = act(g,u),
 * y = Wd a.  Wg, Wu are [W,H]; Wd is [H,W]; all of dtype wd, with block scales
 * sg, su, sd for the MX formats.  x: H doubles.  g, u, a may be NULL.  y: H
 * doubles (overwritten). */
static void expert_mlp(const oracle_cfg *c, const double *x, const void *Wg, const void *Wu,
                       const void *Wd, int wd, const uint8_t *sg, const uint8_t *su, const uint8_t *sd,
                       int W, double *g, double *u, double *a, double *y)
{
    const int H = c->H;
    double *act = (double *)malloc(sizeof(double) * W);
    for (int i = 0; i < W; i++) {
        double gi = 0.0, ui = 0.0;
        for (int h = 0; h < H; h++) {
            gi += wget(Wg, sg, wd, (size_t)i, (size_t)h, (size_t)W, (size_t)H) * x[h];
            ui += wget(Wu, su, wd, (size_t)i, (size_t)h, (size_t)W, (size_t)H) * x[h];
        }
        act[i] = oracle_act(c, gi, ui);
        if (g) g[i] = gi;
        if (u) u[i] = ui;
        if (a) a[i] = act[i];
    }
    for (int h = 0; h < H; h++) {
        double acc = 0.0;
        for (int i = 0; i < W; i++) acc += wget(Wd, sd, wd, (size_t)h, (size_t)i, (size_t)H, (size_t)W) * act[i];
        y[h] = acc;
    }
    free(act);
}

/* ---------------------------------------------------------------- threads */

typedef struct {
    const oracle_cfg *c;
    const void *X;
    int xd;
    const float *Wr, *bias;
    const void *Wg, *Wu, *Wd, *Wgs, *Wus, *Wds;
    int wd;
    const uint8_t *sc[6]; /* MX block scales of Wg, Wu, Wd, Wgs, Wus, Wds */
    const int *tokens;
    int n;
    /* route outputs */
    double *logits, *scores, *biased, *w, *margin;
    int *idx;
    /* forward output */
    double *Y;
    int mode; /* 0 routing, 1 block forward, 2 dense MLP (width S, tensors Wgs/Wus/Wds) */
    int nthreads, tid;
} job;

static int token_of(const job *j, int i) { return j->tokens ? j->tokens[i] : i; }

static void forward_token(const job *j, int i)
{
    const oracle_cfg *c = j->c;
    const int H = c->H, k = c->k, I = c->I;
    const size_t t = (size_t)token_of(j, i);
    int *idx = (int *)malloc(sizeof(int) * k);
    double *w = (double *)malloc(sizeof(double) * k);
    double *x = (double *)malloc(sizeof(double) * H * 3);
    double *ye = x + H, *y = ye + H;

    route_token(c, j->X, j->xd, t, j->Wr, j->bias, NULL, NULL, NULL, idx, w, NULL);
    for (int h = 0; h < H; h++) x[h] = ld(j->X, j->xd, t * H + h);
    for (int h = 0; h < H; h++) y[h] = 0.0;

    const size_t gsz = (size_t)I * H; /* one slice of the stacked gate/up/down */
    const int m = mx(j->wd);
    for (int s = 0; s <= k; s++) {
        /* the k routed experts, then the packed shared expert (slice E, weight 1.0) */
        if (s == k && !c->shared_packed) break;
        const size_t e = s < k ? (size_t)idx[s] : (size_t)c->E;
        const size_t off = wbytes(j->wd, e * gsz), soff = e * gsz / 32;
        expert_mlp(c, x, (const char *)j->Wg + off, (const char *)j->Wu + off,
                   (const char *)j->Wd + off, j->wd, m ? j->sc[0] + soff : NULL,
                   m ? j->sc[1] + soff : NULL, m ? j->sc[2] + soff : NULL, I, NULL, NULL, NULL, ye);
        const double ws = s < k ? w[s] : 1.0;
        for (int h = 0; h < H; h++) y[h] += ws * ye[h];
    }
    if (!c->shared_packed && c->S > 0) {
        expert_mlp(c, x, j->Wgs, j->Wus, j->Wds, j->wd, j->sc[3], j->sc[4], j->sc[5], c->S, NULL, NULL, NULL,
                   ye);
        for (int h = 0; h < H; h++) y[h] += 1.0 * ye[h];
    }
    for (int h = 0; h < H; h++) j->Y[(size_t)i * H + h] = y[h];
    free(x);
    free(w);
    free(idx);
}

static void dense_token(const job *j, int i)
{
    const oracle_cfg *c = j->c;
    const int H = c->H;
    const size_t t = (size_t)token_of(j, i);
    double *x = (double *)malloc(sizeof(double) * H);
    for (int h = 0; h < H; h++) x[h] = ld(j->X, j->xd, t * H + h);
    expert_mlp(c, x, j->Wgs, j->Wus, j->Wds, j->wd, j->sc[3], j->sc[4], j->sc[5], c->S, NULL, NULL, NULL,
               j->Y + (size_t)i * H);
    free(x);
}

static void route_one(const job *j, int i)
{
    const oracle_cfg *c = j->c;
    const size_t E = (size_t)c->E, k = (size_t)c->k;
    route_token(c, j->X, j->xd, (size_t)token_of(j, i), j->Wr, j->bias,
                j->logits ? j->logits + i * E : NULL, j->scores ? j->scores + i * E : NULL,
                j->biased ? j->biased + i * E : NULL, j->idx ? j->idx + i * k : NULL,
                j->w ? j->w + i * k : NULL, j->margin ? j->margin + i : NULL);
}

static void *worker(void *arg)
{
    const job *j = (const job *)arg;
    for (int i = j->tid; i < j->n; i += j->nthreads) {
        if (j->mode == 1)
            forward_token(j, i);
        else if (j->mode == 2)
            dense_token(j, i);
        else
            route_one(j, i);
    }
    return NULL;
}

static int run_jobs(job *proto, int nthreads)
{
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > proto->n) nthreads = proto->n > 0 ? proto->n : 1;
    job *jobs = (job *)malloc(sizeof(job) * nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = *proto;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
    }
    int started = 0;
    for (int t = 1; t < nthreads; t++) {
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) break;
        started = t;
    }
    worker(&jobs[0]);
    for (int t = 1; t <= started; t++) pthread_join(th[t], NULL);
    /* threads that could not be started: run their share here */
    for (int t = started + 1; t < nthreads; t++) worker(&jobs[t]);
    free(th);
    free(jobs);
    return nthreads;
}

static int cfg_ok(const oracle_cfg *c)
{
    return c && c->H > 0 && c->E > 0 && c->k > 0 && c->k <= c->E && c->I >= 0 && c->S >= 0;
}

/* ------------------------------------------------------------- public API */

/* Routing of n tokens (tokens[i], or i when tokens is NULL).
 * Outputs are per listed token: logits/scores/biased [n,E], idx [n,k],
 * w [n,k], margin [n]; any may be NULL.  Returns threads used, or -1. */
int oracle_route(const oracle_cfg *c, const void *X, int x_dtype, const float *Wr,
                 const float *bias, int n, const int *tokens, double *logits, double *scores,
                 double *biased, int *idx, double *w, double *margin, int nthreads)
{
    if (!cfg_ok(c) || !X || !Wr || n < 0) return -1;
    job j;
    memset(&j, 0, sizeof j);
    j.c = c;
    j.X = X;
    j.xd = x_dtype;
    j.Wr = Wr;
    j.bias = bias;
    j.tokens = tokens;
    j.n = n;
    j.logits = logits;
    j.scores = scores;
    j.biased = biased;
    j.idx = idx;
    j.w = w;
    j.margin = margin;
    return run_jobs(&j, nthreads);
}

/* the six MX scale pointers are present for the tensors that are used */
static int scales_ok(const uint8_t *const *sc, int w_dtype, int routed, int shared)
{
    if (!mx(w_dtype)) return 1;
    if (!sc) return 0;
    for (int i = 0; i < 3; i++)
        if ((routed && !sc[i]) || (shared && !sc[3 + i])) return 0;
    return 1;
}

/* Full block output for n tokens: Y [n,H] doubles.  Expert tensors: Wg, Wu
 * [E',I,H], Wd [E',H,I] with E' = E (+1 when packed), dtype w_dtype; shared
 * tensors Wgs, Wus [S,H], Wds [H,S] (ignored when packed or S == 0).  MX
 * dtypes: scales[6] = block scales of Wg, Wu, Wd, Wgs, Wus, Wds ([E', H/32, I],
 * [E', H/32, I], [E', I/32, H], [H/32, S], [H/32, S], [S/32, H]); else NULL.
 * Returns threads used, or -1. */
int oracle_forward(const oracle_cfg *c, const void *X, int x_dtype, const float *Wr,
                   const float *bias, const void *Wg, const void *Wu, const void *Wd,
                   const void *Wgs, const void *Wus, const void *Wds, int w_dtype,
                   const uint8_t *const *scales, int n, const int *tokens, double *Y, int nthreads)
{
    if (!cfg_ok(c) || !X || !Wr || !Wg || !Wu || !Wd || !Y || n < 0) return -1;
    if (!c->shared_packed && c->S > 0 && (!Wgs || !Wus || !Wds)) return -1;
    if (!scales_ok(scales, w_dtype, 1, !c->shared_packed && c->S > 0)) return -1;
    job j;
    memset(&j, 0, sizeof j);
    j.c = c;
    j.X = X;
    j.xd = x_dtype;
    j.Wr = Wr;
    j.bias = bias;
    j.Wg = Wg;
    j.Wu = Wu;
    j.Wd = Wd;
    j.Wgs = Wgs;
    j.Wus = Wus;
    j.Wds = Wds;
    j.wd = w_dtype;
    if (mx(w_dtype))
        for (int i = 0; i < 6; i++) j.sc[i] = scales[i];
    j.tokens = tokens;
    j.n = n;
    j.Y = Y;
    j.mode = 1;
    return run_jobs(&j, nthreads);
}

/* Dense MLP of width c->S (router and experts unused) for n tokens: Y [n,H]
 * doubles.  Wg, Wu: [S,H]; Wd: [H,S]; dtype w_dtype, MX scales[3] of Wg, Wu,
 * Wd or NULL.  Returns threads used, or -1. */
int oracle_dense(const oracle_cfg *c, const void *X, int x_dtype, const void *Wg, const void *Wu,
                 const void *Wd, int w_dtype, const uint8_t *const *scales, int n, const int *tokens,
                 double *Y, int nthreads)
{
    if (!c || c->H <= 0 || c->S <= 0 || !X || !Wg || !Wu || !Wd || !Y || n < 0) return -1;
    if (!scales_ok(scales, w_dtype, 1, 0)) return -1;
    job j;
    memset(&j, 0, sizeof j);
    j.c = c;
    j.X = X;
    j.xd = x_dtype;
    j.Wgs = Wg;
    j.Wus = Wu;
    j.Wds = Wd;
    j.wd = w_dtype;
    if (mx(w_dtype))
        for (int i = 0; i < 3; i++) j.sc[3 + i] = scales[i];
    j.tokens = tokens;
    j.n = n;
    j.Y = Y;
    j.mode = 2;
    return run_jobs(&j, nthreads);
}

/* RMSNorm of one row of H values: y_h = x_h / sqrt(mean_h x_h^2 + eps) * g_h,
 * g_h = w_h (gemma = 0) or 1 + w_h (gemma = 1).  Returns 0, or -1. */
int oracle_rmsnorm(const double *x, int H, const double *w, double eps, int gemma, double *y)
{
    if (!x || !w || !y || H <= 0 || eps < 0.0) return -1;
    double ss = 0.0;
    for (int h = 0; h < H; h++) ss += x[h] * x[h];
    const double r = sqrt(ss / (double)H + eps);
    for (int h = 0; h < H; h++) y[h] = x[h] / r * (gemma ? 1.0 + w[h] : w[h]);
    return 0;
}

/* One expert MLP of width W on one token row x (H values of x_dtype), for
 * checking intermediate values: g, u, a [W] and y [H] doubles (g, u, a may be
 * NULL).  Wg, Wu: [W,H]; Wd: [H,W]; dtype w_dtype, MX scales[3] of Wg, Wu, Wd
 * or NULL. */
int oracle_expert(const oracle_cfg *c, const void *x, int x_dtype, const void *Wg,
                  const void *Wu, const void *Wd, int w_dtype, const uint8_t *const *scales, int W,
                  double *g, double *u, double *a, double *y)
{
    if (!c || c->H <= 0 || !x || !Wg || !Wu || !Wd || !y || W <= 0) return -1;
    if (!scales_ok(scales, w_dtype, 1, 0)) return -1;
    double *xd = (double *)malloc(sizeof(double) * c->H);
    for (int h = 0; h < c->H; h++) xd[h] = ld(x, x_dtype, (size_t)h);
    const int m = mx(w_dtype);
    expert_mlp(c, xd, Wg, Wu, Wd, w_dtype, m ? scales[0] : NULL, m ? scales[1] : NULL, m ? scales[2] : NULL, W,
               g, u, a, y);
    free(xd);
    return 0;
}

/* Decoded value of one MX element code (dtype OR_MXFP8: a byte; OR_MXFP4: a
 * nibble) times the E8M0 scale code, for checking the decoders. */
double oracle_mx_value(int w_dtype, int code, int scale)
{
    const double sc = e8m0((uint8_t)scale);
    if (w_dtype == OR_MXFP8) return sc * e4m3((uint8_t)code);
    if (w_dtype == OR_MXFP4) return sc * e2m1((uint8_t)(code & 15));
    return NAN;
}
