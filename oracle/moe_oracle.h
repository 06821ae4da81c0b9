/*
 * Reference oracle for the int4 routed-MoE FFN step -- TEST INFRASTRUCTURE.
 *
 * A plain, slow, double-precision CPU statement of what the step computes.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it; the GPU library never does, and the two share no code.
 *
 * Sources (page, section):
 *  - "25GB 内存上运行 GLM 5.2 744B" (reader.mx), section 11 "MoE 路由与专家执行":
 *    sigmoid(logit) + correction bias selects the top-K; the weight is the
 *    un-biased sigmoid times routed_scale; greedy K-pass argmax, strict '>',
 *    so the lowest index wins a tie; SwiGLU expert h = silu(g) * u, d = W_d h;
 *    weighted accumulate of the expert outputs.
 *  - same page, section 06 "从 FP8 到 int4": row-wise symmetric int4, qmax 7,
 *    s = max(amax/7, 1e-8), q = clip(rint(w/s), -8, 7); stored q+8, element
 *    2j in the low nibble, 2j+1 in the high nibble; row stride ceil(I/2)
 *    bytes, pad nibble 8; one float32 scale per output row (".qs").
 *  - same page, section 04 "手写的基础数学": RMSNorm and SiLU.
 *  - same page, section 03 (the OLMoE engine): int8 expert weights, one signed
 *    byte per value and one float32 scale per row (quantize_rows, bits = 8).
 *  - Edge0 article, section 三: int4 affine with group size 64 (1.77 MB per
 *    expert of the 35B-class model, group scales included).
 *  - Edge0 article (magicnetworld.com), section 七 "路由数学": renormalised
 *    sigmoid weights w_i = s * sigma_i / (sum_{j in S} sigma_j + 1e-20); the
 *    softmax-top-k family (g = softmax(logits), top-K of g, w_i = g_i / sum_S g)
 *    and group-limited selection for the sigmoid family (groups ranked by the
 *    sum of their two best selection scores, the best topk_group kept, the
 *    rest masked to -inf, then top-K among the survivors).
 *  - reader.mx page, section 03 (the OLMoE engine's moe()): softmax over the E
 *    logits, greedy top-K by strict '>', weight = the probability itself.
 *  - GLM-5.2 operator breakdown (devpress.csdn.net), section 2.3 and stage
 *    "Step 6 (MoE)" 6a-6d: output = sum of routed outputs + shared expert.
 *
 * Every floating-point step is done in double, except the offline quantiser
 * oracle_quantize_int4, which follows the page's float32 arithmetic because
 * its output bytes are what the pages define.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int H;            /* hidden size */
    int E;            /* routed experts */
    int K;            /* top-k */
    int I;            /* routed expert intermediate size */
    int n_shared;     /* 0 or 1 */
    int I_shared;     /* shared expert intermediate size */
    int n_group;      /* expert groups (E % n_group == 0); > 1 only with the sigmoid score */
    int norm_topk;    /* 1: renormalise the selected weights */
    int prenorm_residual; /* 1: y = x + moe(rmsnorm(x)) */
    double routed_scale;
    double rms_eps;
    int topk_group;   /* groups kept when n_group > 1 (1..n_group) */
    int score_func;   /* ORACLE_SCORE_SIGMOID or ORACLE_SCORE_SOFTMAX */
    int expert_format;   /* routed experts: ORACLE_FORMAT_INT4 or ORACLE_FORMAT_INT8 */
    int shared_format;   /* shared expert: the same choice */
} oracle_cfg;

#define ORACLE_FORMAT_INT4 0     /* section 06: two values per byte, q + 8, low nibble first */
#define ORACLE_FORMAT_INT8 1     /* section 03 (OLMoE engine): one signed byte per value */
#define ORACLE_FORMAT_G64 2      /* Edge0 article section 三: int4 affine, group size 64 */

#define ORACLE_SCORE_SIGMOID 0   /* sigma = sigmoid(logit); selection by sigma + bias */
#define ORACLE_SCORE_SOFTMAX 1   /* g = softmax(logits); selection by g; bias unused */

typedef struct {
    const float *router_w;            /* [E, H] */
    const float *router_b;            /* [E] */
    const uint8_t *const *slab;       /* E pointers: gate | up | down packed bytes */
    const float *const *scale;        /* E pointers: sg[I] | su[I] | sd[H] */
    const uint8_t *sh_slab;           /* shared expert, same layout with I_shared */
    const float *sh_scale;
} oracle_layer;

/* int4 unpack of n values from one packed row: q[i] = nibble - 8. */
void oracle_unpack_int4(const uint8_t *row, int n, int *q);

/* Per-row symmetric int4 codes of a float32 matrix [O, I] (section 06), computed
 * in float32 because the stored bytes and scales are what the page defines. */
void oracle_quantize_int4(const float *w, int O, int I, uint8_t *q4, float *scale);

/* Per-row symmetric int8 codes of a float32 matrix [O, I] (section 03, the
 * OLMoE engine's 8-bit weights), computed in float32 like the int4 quantiser. */
void oracle_quantize_int8(const float *w, int O, int I, int8_t *q, float *scale);

/* oracle_expert for any weight format (ORACLE_FORMAT_*); the int8 slab is
 * gate [I, H] | up [I, H] | down [H, I] signed bytes with the same scales.
 * ORACLE_FORMAT_G64: the int4 slab layout with unsigned nibbles u in [0, 15]
 * (element 2j low), and `scale` is not float32 but float16 pairs (s, b), one
 * per 64 consecutive inputs of a row: gate [I][H/64] | up [I][H/64] |
 * down [H][I/64], W[o,i] = s * u + b of the row's group i / 64 (H, I multiples
 * of 64).  Read as uint16 bit patterns and widened exactly. */
void oracle_expert_fmt(int H, int I, int format, const uint8_t *slab, const float *scale,
                       const double *x, double *d_out, double *h_out);

double oracle_silu(double v);

/* RMSNorm with unit weight: out = x / sqrt(mean(x^2) + eps). */
void oracle_rmsnorm(const double *x, int H, double eps, double *out);

/* One SwiGLU expert on one token: d[H] = W_d (silu(W_g x) * (W_u x)). */
void oracle_expert(int H, int I, const uint8_t *slab, const float *scale,
                   const double *x, double *d_out, double *h_out /* nullable, [I] */);

/* Router for one token.  Returns 0, or -1 on an invalid config.
 * idx[K] in descending selection-score order, w[K] routing weights,
 * *margin = c_(K) - c_(K+1) (+inf when none is left), and with groups the
 * smaller of that and gs_(topk_group) - gs_(topk_group+1) over the group
 * scores; scores (nullable) [3*E]: logits | sigmoid (softmax probability) |
 * selection score (-inf outside the kept groups). */
int oracle_route(const oracle_cfg *c, const float *router_w, const float *router_b,
                 const double *x, int *idx, double *w, double *margin, double *scores);

/* Routing weights of a given selection (used to re-score a GPU selection). */
int oracle_weights_for(const oracle_cfg *c, const float *router_w, const double *x,
                       const int *idx, double *w);

/* One token through one layer.  forced_idx (nullable) replaces the top-k
 * selection.  y[H]; idx[K], w[K], margin outputs may be NULL. */
int oracle_moe_token(const oracle_cfg *c, const oracle_layer *L, const double *x,
                     const int *forced_idx, double *y, int *idx, double *w, double *margin);

/* T tokens of float32 input through one layer (loops oracle_moe_token). */
int oracle_moe_forward(const oracle_cfg *c, const oracle_layer *L, const float *x, int T,
                       double *y, int *idx, double *w, double *margin);

/* Threads an OpenMP build would use (1 without OpenMP). */
int oracle_threads(void);
void oracle_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
