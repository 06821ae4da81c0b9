/*
 * Reference oracle for the int4 routed-MoE FFN step -- TEST INFRASTRUCTURE.
 * Plain double-precision C; see moe_oracle.h for the sources each step
 * follows.  Nothing here is blocked, fused or reordered beyond the plain
 * definitions; OpenMP (when enabled) only splits independent output rows.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the following calls (n >= 1); used to time the oracle on one core. */
void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Section 06: element 2j is the low nibble of byte j, 2j+1 the high nibble;
 * the stored nibble is q + 8. */
static int nibble_at(const uint8_t *row, int i) {
    uint8_t b = row[i >> 1];
    int v = (i & 1) ? (b >> 4) : (b & 15);
    return v - 8;
}

void oracle_unpack_int4(const uint8_t *row, int n, int *q) {
    for (int i = 0; i < n; i++) q[i] = nibble_at(row, i);
}

/* Scale of one row for a symmetric signed code with largest code qmax, in
 * float32 as the pages define it: the row's peak magnitude over qmax, floored
 * at 1e-8 so that an all-zero row keeps a finite, non-zero scale. */
static float sym_row_scale(const float *row, int n, int qmax) {
    float peak = 0.f;
    for (int i = 0; i < n; i++) peak = fmaxf(peak, fabsf(row[i]));
    return fmaxf(peak / (float)qmax, 1e-8f);
}

/* The code of v under scale s: v / s rounded to the nearest integer (ties to
 * even, rintf in the default rounding mode), held inside [lo, hi]; NaN -> lo. */
static int sym_code(float v, float s, int lo, int hi) {
    const float c = rintf(v / s);
    if (!(c > (float)lo)) return lo;
    if (c > (float)hi) return hi;
    return (int)c;
}

/* int4 per-row quantiser of the reader.mx page, section 06 "从 FP8 到 int4":
 * codes in [-8, 7] under sym_row_scale(row, 7), stored as code + 8 with element
 * 2j in the low nibble of byte j; an odd row's last byte is padded with code 0. */
void oracle_quantize_int4(const float *w, int O, int I, uint8_t *q4, float *scale) {
    const int stride = (I + 1) / 2;
    memset(q4, 0x88, (size_t)O * (size_t)stride);   /* every nibble holds code 0 */
    for (int o = 0; o < O; o++) {
        const float *row = w + (int64_t)o * I;
        uint8_t *dst = q4 + (int64_t)o * stride;
        const float s = sym_row_scale(row, I, 7);
        scale[o] = s;
        for (int i = 0; i < I; i++) {
            const unsigned nib = (unsigned)(sym_code(row[i], s, -8, 7) + 8);
            const unsigned shift = 4u * (unsigned)(i & 1);
            dst[i >> 1] = (uint8_t)((dst[i >> 1] & ~(15u << shift)) | (nib << shift));
        }
    }
}

double oracle_silu(double v) { return v / (1.0 + exp(-v)); }

/* Section 04 RMSNorm with unit weight. */
void oracle_rmsnorm(const double *x, int H, double eps, double *out) {
    double ms = 0.0;
    for (int i = 0; i < H; i++) ms += x[i] * x[i];
    double r = 1.0 / sqrt(ms / H + eps);
    for (int i = 0; i < H; i++) out[i] = x[i] * r;
}

/* out[o] = scale[o] * sum_i q[o,i] * v[i] over one packed [O, ceil(n/2)] matrix. */
static void int4_matvec(const uint8_t *q4, const float *scale, int O, int n,
                        const double *v, double *out) {
    const int rb = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int o = 0; o < O; o++) {
        const uint8_t *row = q4 + (int64_t)o * rb;
        double acc = 0.0;
        for (int i = 0; i < n; i++) acc += (double)nibble_at(row, i) * v[i];
        out[o] = (double)scale[o] * acc;
    }
}

/* out[o] = scale[o] * sum_i q[o,i] * v[i] over one int8 [O, n] matrix (row stride n bytes). */
static void int8_matvec(const uint8_t *q8, const float *scale, int O, int n,
                        const double *v, double *out) {
#pragma omp parallel for schedule(static)
    for (int o = 0; o < O; o++) {
        const int8_t *row = (const int8_t *)(q8 + (int64_t)o * n);
        double acc = 0.0;
        for (int i = 0; i < n; i++) acc += (double)row[i] * v[i];
        out[o] = (double)scale[o] * acc;
    }
}

/* int8 per-row quantiser of the reader.mx page's OLMoE engine (section 03,
 * 8-bit codes): codes in [-128, 127] under sym_row_scale(row, 127), one signed
 * byte per value. */
void oracle_quantize_int8(const float *w, int O, int I, int8_t *q, float *scale) {
    for (int o = 0; o < O; o++) {
        const float *row = w + (int64_t)o * I;
        int8_t *dst = q + (int64_t)o * I;
        scale[o] = sym_row_scale(row, I, 127);
        for (int i = 0; i < I; i++) dst[i] = (int8_t)sym_code(row[i], scale[o], -128, 127);
    }
}

/* IEEE binary16 bit pattern -> double (exact). */
static double half_to_double(uint16_t h) {
    const int sgn = h >> 15, ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 0) v = ldexp((double)man, -24);                      /* zero, subnormal */
    else if (ex == 31) v = man ? NAN : INFINITY;
    else v = ldexp((double)(man + 1024), ex - 25);
    return sgn ? -v : v;
}

/* out[o] = sum_i (s_{o,i/64} u[o,i] + b_{o,i/64}) v[i] over one affine-int4 [O, n]
 * matrix: packed rows of n/2 bytes, (s, b) float16 pairs [O][n/64]. */
static void g64_matvec(const uint8_t *q4, const uint16_t *sb, int O, int n, const double *v, double *out) {
    const int rb = n / 2, ng = n / 64;
#pragma omp parallel for schedule(static)
    for (int o = 0; o < O; o++) {
        const uint8_t *row = q4 + (int64_t)o * rb;
        double acc = 0.0;
        for (int i = 0; i < n; i++) {
            const int u = (i & 1) ? (row[i >> 1] >> 4) : (row[i >> 1] & 15);
            const uint16_t *p = sb + 2 * ((int64_t)o * ng + i / 64);
            acc += (half_to_double(p[0]) * u + half_to_double(p[1])) * v[i];
        }
        out[o] = acc;
    }
}

/* Section 11 expert in either weight format: g = W_g x, u = W_u x,
 * h = silu(g) * u, d = W_d h.  int8 slab: gate [I, H] | up [I, H] | down [H, I]
 * bytes, signed, one float32 scale per output row as for int4. */
void oracle_expert_fmt(int H, int I, int format, const uint8_t *slab, const float *scale,
                       const double *x, double *d_out, double *h_out) {
    if (format == ORACLE_FORMAT_G64) {
        const int64_t rbH = H / 2;
        const uint16_t *sb = (const uint16_t *)scale;
        double *g = (double *)malloc(sizeof(double) * I);
        double *u = (double *)malloc(sizeof(double) * I);
        double *h = (double *)malloc(sizeof(double) * I);
        g64_matvec(slab, sb, I, H, x, g);
        g64_matvec(slab + (int64_t)I * rbH, sb + 2 * (int64_t)I * (H / 64), I, H, x, u);
        for (int i = 0; i < I; i++) h[i] = oracle_silu(g[i]) * u[i];
        g64_matvec(slab + 2 * (int64_t)I * rbH, sb + 4 * (int64_t)I * (H / 64), H, I, h, d_out);
        if (h_out) memcpy(h_out, h, sizeof(double) * I);
        free(g); free(u); free(h);
        return;
    }
    if (format != ORACLE_FORMAT_INT8) {
        oracle_expert(H, I, slab, scale, x, d_out, h_out);
        return;
    }
    const uint8_t *qg = slab, *qu = slab + (int64_t)I * H, *qd = slab + 2 * (int64_t)I * H;
    const float *sg = scale, *su = scale + I, *sd = scale + 2 * I;
    double *g = (double *)malloc(sizeof(double) * I);
    double *u = (double *)malloc(sizeof(double) * I);
    double *h = (double *)malloc(sizeof(double) * I);
    int8_matvec(qg, sg, I, H, x, g);
    int8_matvec(qu, su, I, H, x, u);
    for (int i = 0; i < I; i++) h[i] = oracle_silu(g[i]) * u[i];
    int8_matvec(qd, sd, H, I, h, d_out);
    if (h_out) memcpy(h_out, h, sizeof(double) * I);
    free(g); free(u); free(h);
}

/* Section 11 expert: g = W_g x, u = W_u x, h = silu(g) * u, d = W_d h. */
void oracle_expert(int H, int I, const uint8_t *slab, const float *scale,
                   const double *x, double *d_out, double *h_out) {
    const int64_t rbH = (H + 1) / 2;
    const uint8_t *qg = slab;
    const uint8_t *qu = slab + (int64_t)I * rbH;
    const uint8_t *qd = slab + 2 * (int64_t)I * rbH;
    const float *sg = scale, *su = scale + I, *sd = scale + 2 * I;
    double *g = (double *)malloc(sizeof(double) * I);
    double *u = (double *)malloc(sizeof(double) * I);
    double *h = (double *)malloc(sizeof(double) * I);
    int4_matvec(qg, sg, I, H, x, g);
    int4_matvec(qu, su, I, H, x, u);
    for (int i = 0; i < I; i++) h[i] = oracle_silu(g[i]) * u[i];
    int4_matvec(qd, sd, H, I, h, d_out);
    if (h_out) memcpy(h_out, h, sizeof(double) * I);
    free(g); free(u); free(h);
}

typedef struct { double c; int e; } scored;

/* Order: larger selection score first; on equal scores the lower index first
 * (what a strict '>' scan in ascending index order produces). */
static int by_score_desc(const void *a, const void *b) {
    const scored *p = (const scored *)a, *q = (const scored *)b;
    if (p->c > q->c) return -1;
    if (p->c < q->c) return 1;
    return (p->e > q->e) - (p->e < q->e);
}

static int cfg_ok(const oracle_cfg *c) {
    if (!c || c->H <= 0 || c->E <= 0 || c->K <= 0 || c->K > c->E || c->I <= 0) return 0;
    if (!(c->n_shared == 0 || (c->n_shared == 1 && c->I_shared > 0))) return 0;
    if (c->score_func != ORACLE_SCORE_SIGMOID && c->score_func != ORACLE_SCORE_SOFTMAX) return 0;
    if (c->expert_format < ORACLE_FORMAT_INT4 || c->expert_format > ORACLE_FORMAT_G64 ||
        c->shared_format < ORACLE_FORMAT_INT4 || c->shared_format > ORACLE_FORMAT_G64) return 0;
    if ((c->expert_format == ORACLE_FORMAT_G64 || (c->n_shared && c->shared_format == ORACLE_FORMAT_G64)) &&
        (c->H % 64 || c->I % 64 || (c->n_shared && c->I_shared % 64))) return 0;
    if (c->n_group < 1 || c->E % c->n_group != 0) return 0;
    if (c->n_group > 1) {
        if (c->score_func != ORACLE_SCORE_SIGMOID) return 0;
        if (c->topk_group < 1 || c->topk_group > c->n_group) return 0;
        if (c->K > c->topk_group * (c->E / c->n_group)) return 0;
    }
    return 1;
}

/* Per-expert scores.  Sigmoid family: sig = sigmoid(logit), selection score
 * sig + bias.  Softmax family: sig = softmax(logits) (shifted by the largest
 * logit), selection score sig; the bias is not used. */
static void router_scores(const oracle_cfg *c, const float *W, const float *b,
                          const double *x, double *logit, double *sig, double *choice) {
#pragma omp parallel for schedule(static)
    for (int e = 0; e < c->E; e++) {
        const float *wr = W + (int64_t)e * c->H;
        double acc = 0.0;
        for (int h = 0; h < c->H; h++) acc += (double)wr[h] * x[h];
        logit[e] = acc;
    }
    if (c->score_func == ORACLE_SCORE_SOFTMAX) {
        double m = -INFINITY, z = 0.0;
        for (int e = 0; e < c->E; e++) m = logit[e] > m ? logit[e] : m;
        for (int e = 0; e < c->E; e++) z += exp(logit[e] - m);
        for (int e = 0; e < c->E; e++) {
            sig[e] = exp(logit[e] - m) / z;
            choice[e] = sig[e];
        }
    } else {
        for (int e = 0; e < c->E; e++) {
            sig[e] = 1.0 / (1.0 + exp(-logit[e]));
            choice[e] = sig[e] + (double)b[e];
        }
    }
}

/* Group-limited selection (n_group > 1): group g holds experts
 * [g E/n_group, (g+1) E/n_group); its score is the sum of its two best
 * selection scores (one when a group has one expert).  The topk_group best
 * groups are kept (ties: lower group first) and every expert of the other
 * groups gets -inf.  Returns gs_(topk_group) - gs_(topk_group+1), +inf when
 * every group is kept. */
static double mask_groups(const oracle_cfg *c, double *choice) {
    const int G = c->n_group, m = c->E / c->n_group;
    if (G <= 1) return INFINITY;
    scored *gs = (scored *)malloc(sizeof(scored) * G);
    for (int g = 0; g < G; g++) {
        double b1 = -INFINITY, b2 = -INFINITY;
        for (int i = 0; i < m; i++) {
            const double v = choice[g * m + i];
            if (v > b1) { b2 = b1; b1 = v; }
            else if (v > b2) b2 = v;
        }
        gs[g].c = m > 1 ? b1 + b2 : b1;
        gs[g].e = g;
    }
    qsort(gs, G, sizeof(scored), by_score_desc);
    for (int r = c->topk_group; r < G; r++)
        for (int i = 0; i < m; i++) choice[gs[r].e * m + i] = -INFINITY;
    const double gm = c->topk_group < G ? gs[c->topk_group - 1].c - gs[c->topk_group].c : INFINITY;
    free(gs);
    return gm;
}

/* Weights of the selection idx[K]: w_k = s * sig_k / (sum_S sig + 1e-20) for the
 * sigmoid family, s * g_k / sum_S g for the softmax family (norm_topk); s * sig_k
 * (s * g_k) without renormalisation. */
static void weights_of(const oracle_cfg *c, const double *sig, const int *idx, double *w) {
    double den = 0.0;
    for (int k = 0; k < c->K; k++) den += sig[idx[k]];
    if (c->score_func == ORACLE_SCORE_SIGMOID) den += 1e-20;
    for (int k = 0; k < c->K; k++)
        w[k] = c->norm_topk ? c->routed_scale * sig[idx[k]] / den
                            : c->routed_scale * sig[idx[k]];
}

int oracle_route(const oracle_cfg *c, const float *router_w, const float *router_b,
                 const double *x, int *idx, double *w, double *margin, double *scores) {
    if (!cfg_ok(c)) return -1;
    const int E = c->E, K = c->K;
    double *logit = (double *)malloc(sizeof(double) * 3 * E);
    double *sig = logit + E, *choice = logit + 2 * E;
    router_scores(c, router_w, router_b, x, logit, sig, choice);
    const double gmargin = mask_groups(c, choice);
    scored *s = (scored *)malloc(sizeof(scored) * E);
    for (int e = 0; e < E; e++) { s[e].c = choice[e]; s[e].e = e; }
    qsort(s, E, sizeof(scored), by_score_desc);
    for (int k = 0; k < K; k++) idx[k] = s[k].e;
    if (margin) {
        double mg = (K < E && s[K].c > -INFINITY) ? s[K - 1].c - s[K].c : INFINITY;
        *margin = gmargin < mg ? gmargin : mg;
    }
    if (w) weights_of(c, sig, idx, w);
    if (scores) memcpy(scores, logit, sizeof(double) * 3 * E);
    free(s);
    free(logit);
    return 0;
}

int oracle_weights_for(const oracle_cfg *c, const float *router_w, const double *x,
                       const int *idx, double *w) {
    if (!cfg_ok(c)) return -1;
    double *logit = (double *)malloc(sizeof(double) * 3 * c->E);
    double *sig = logit + c->E, *choice = logit + 2 * c->E;
    float *zero_b = (float *)calloc(c->E, sizeof(float));   /* the bias does not enter weights */
    router_scores(c, router_w, zero_b, x, logit, sig, choice);
    free(zero_b);
    for (int k = 0; k < c->K; k++)
        if (idx[k] < 0 || idx[k] >= c->E) { free(logit); return -1; }
    weights_of(c, sig, idx, w);
    free(logit);
    return 0;
}

int oracle_moe_token(const oracle_cfg *c, const oracle_layer *L, const double *x,
                     const int *forced_idx, double *y, int *idx_out, double *w_out,
                     double *margin) {
    if (!cfg_ok(c)) return -1;
    const int H = c->H, K = c->K;
    double *xin = (double *)malloc(sizeof(double) * H);
    double *d = (double *)malloc(sizeof(double) * H);
    double *acc = (double *)calloc(H, sizeof(double));
    int *idx = (int *)malloc(sizeof(int) * K);
    double *w = (double *)malloc(sizeof(double) * K);
    int rc = 0;

    if (c->prenorm_residual) oracle_rmsnorm(x, H, c->rms_eps, xin);
    else memcpy(xin, x, sizeof(double) * H);

    double mg = INFINITY;
    if (forced_idx) {
        memcpy(idx, forced_idx, sizeof(int) * K);
        rc = oracle_weights_for(c, L->router_w, xin, idx, w);
    } else {
        rc = oracle_route(c, L->router_w, L->router_b, xin, idx, w, &mg, NULL);
    }
    if (rc == 0) {
        /* routed experts in selection order, then the shared expert (weight 1) */
        for (int k = 0; k < K && rc == 0; k++) {
            const uint8_t *slab = L->slab[idx[k]];
            const float *scale = L->scale[idx[k]];
            if (!slab || !scale) { rc = -2; break; }
            oracle_expert_fmt(H, c->I, c->expert_format, slab, scale, xin, d, NULL);
            for (int h = 0; h < H; h++) acc[h] += w[k] * d[h];
        }
        if (rc == 0 && c->n_shared) {
            oracle_expert_fmt(H, c->I_shared, c->shared_format, L->sh_slab, L->sh_scale, xin, d, NULL);
            for (int h = 0; h < H; h++) acc[h] += d[h];
        }
        if (rc == 0) {
            for (int h = 0; h < H; h++) y[h] = c->prenorm_residual ? x[h] + acc[h] : acc[h];
            if (idx_out) memcpy(idx_out, idx, sizeof(int) * K);
            if (w_out) memcpy(w_out, w, sizeof(double) * K);
            if (margin) *margin = mg;
        }
    }
    free(xin); free(d); free(acc); free(idx); free(w);
    return rc;
}

int oracle_moe_forward(const oracle_cfg *c, const oracle_layer *L, const float *x, int T,
                       double *y, int *idx, double *w, double *margin) {
    if (!cfg_ok(c) || T < 0) return -1;
    double *xd = (double *)malloc(sizeof(double) * c->H);
    int rc = 0;
    for (int t = 0; t < T && rc == 0; t++) {
        for (int h = 0; h < c->H; h++) xd[h] = (double)x[(int64_t)t * c->H + h];
        rc = oracle_moe_token(c, L, xd, NULL, y + (int64_t)t * c->H,
                              idx ? idx + (int64_t)t * c->K : NULL,
                              w ? w + (int64_t)t * c->K : NULL,
                              margin ? margin + t : NULL);
    }
    free(xd);
    return rc;
}
