/*
 * moe.h -- C ABI of the GB300 int4 routed-MoE FFN step.
 *
 * One call computes, for T tokens x[T,H] (float32, device memory),
 *
 *     y[t] = sum_{k<K} w[t,k] * FFN_{e[t,k]}(x[t]) + FFN_shared(x[t])
 *
 * where FFN_e(v) = W_d,e (silu(W_g,e v) * (W_u,e v)) is a SwiGLU expert whose
 * three matrices are row-quantised int4, and (e[t,.], w[t,.]) is the router's
 * choice.  Sources, by page and section:
 *
 *  - Router ("25GB 内存上运行 GLM 5.2 744B", reader.mx, section 11 "MoE 路由与
 *    专家执行"): logit = W_r x (float32, W_r [E,H]); sigma = sigmoid(logit);
 *    the top-K of sigma + bias[e] (e_score_correction_bias) is selected; the
 *    weight uses the un-biased sigma, times routed_scaling_factor.  A tie is
 *    won by the lower expert index; the K choices come out in descending
 *    score order.
 *  - Renormalisation (Edge0 article, magicnetworld.com, section 七 "路由数学",
 *    sigmoid family): w = s * sigma / (sum_{selected} sigma + 1e-20).
 *  - Routing variants (same section): group-limited selection for the sigmoid
 *    family (n_group > 1: groups ranked by the sum of their two best selection
 *    scores, the best topk_group kept, every expert of the other groups masked
 *    to -inf before the top-K; a group tie is won by the lower group index);
 *    the softmax family (score_func = MOE_SCORE_SOFTMAX: g = softmax(logits),
 *    top-K of g, the bias unused, w = s * g / sum_{selected} g, or s * g
 *    without renormalisation as in the OLMoE engine of the reader.mx page,
 *    section 03).
 *  - Expert format (reader.mx page, section 06 "从 FP8 到 int4"): each row of a
 *    matrix [O, n] is ceil(n/2) bytes, element 2j in the low nibble of byte j
 *    and 2j+1 in the high nibble, stored as q+8 with q in [-8, 7]; one float32
 *    scale per output row, so W[o,i] = (nibble - 8) * scale[o].
 *  - Composition (GLM-5.2 operator breakdown, devpress.csdn.net, "Step 6 (MoE)"
 *    sub-steps 6a-6d): 8 routed experts plus one always-active shared expert,
 *    whose output is added with weight 1.
 *  - Optional pre-norm + residual (reader.mx page, section 04): with
 *    MOE_FLAG_PRENORM_RESIDUAL the call computes y = x + moe(rmsnorm(x)),
 *    rmsnorm(x) = x / sqrt(mean(x^2) + rms_eps) with unit weight.
 *
 * Everything runs on the current CUDA device, on the caller's stream, with
 * no host synchronisation (except moe_forward_host, which is synchronous by
 * design).  There is no CPU fallback: every failure is a status code.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4

/* y = x + moe(rmsnorm(x)) instead of y = moe(x). */
#define MOE_FLAG_PRENORM_RESIDUAL 1u
/* Record the timeline of every T == 1 call on the single-kernel decode path
 * (see moe_trace_read); results are identical with and without it. */
#define MOE_FLAG_TRACE 2u
/* T > 1 calls use the CUDA-core batched kernels (exact f32 arithmetic) even
 * where the tensor-core kernels apply (for comparisons at small T). */
#define MOE_FLAG_CUDA_CORES 4u

/* Checked build of the path (bounds and invariants, in place of a memory
 * checker): every call on the handle runs one more kernel after the step that
 * verifies the call's routing and buckets -- each top-K index in [0, E) and
 * distinct within its token, each routing weight finite, and where the call
 * built buckets (T > 1, or T == 1 off the single-kernel decode path) counts
 * that are the running differences of the offsets, every pair of an expert the
 * handle computes at a position within its expert's range with perm and inv
 * inverse to each other there, and every other pair without a position.  A
 * failed check sets MOE_DEVICE_ERR_CHECK in the device error word (see
 * moe_device_error); the output of that call is not to be trusted. */
#define MOE_FLAG_DEBUG_CHECKS 8u

/* Bits of the device error word (moe_device_error). */
#define MOE_DEVICE_ERR_GRID 8u     /* a grid-wide wait of the decode kernel ran out */
#define MOE_DEVICE_ERR_CHECK 16u   /* a check of MOE_FLAG_DEBUG_CHECKS failed */
#define MOE_DEVICE_ERR_TC 32u      /* a pipeline wait of the tcgen05 expert kernel ran out */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = 1,      /* bad argument or config; nothing was launched */
    MOE_ERR_CUDA = 2,         /* a CUDA call failed; see moe_last_error() */
    MOE_ERR_NOMEM = 3,        /* device allocation failed */
    MOE_ERR_UNSUPPORTED = 4   /* well-formed but outside what the kernels cover */
} moe_status;

typedef struct moe_config {
    int32_t hidden;        /* H: multiple of 32, 32..16384 */
    int32_t n_experts;     /* E: 1..1024 */
    int32_t top_k;         /* K: 1..min(E, 32) */
    int32_t moe_inter;     /* I: multiple of 32, 32..16384 */
    int32_t n_shared;      /* 0 or 1 */
    int32_t shared_inter;  /* I_sh: multiple of 32 when n_shared == 1 */
    int32_t n_group;       /* expert groups: 1..32, divides n_experts; > 1 only with the sigmoid score */
    int32_t norm_topk;     /* 1: renormalise the selected weights (see above); 0: w = s * sigma */
    float routed_scale;    /* s, routed_scaling_factor */
    float rms_eps;         /* used with MOE_FLAG_PRENORM_RESIDUAL */
    uint32_t flags;        /* MOE_FLAG_* */
    int32_t topk_group;    /* groups kept when n_group > 1: 1..n_group, with
                              top_k <= topk_group * n_experts / n_group; ignored when n_group == 1 */
    int32_t score_func;    /* MOE_SCORE_SIGMOID (0) or MOE_SCORE_SOFTMAX (1) */
    int32_t expert_format; /* routed experts: MOE_FORMAT_INT4 (0), MOE_FORMAT_INT8 (1) or MOE_FORMAT_G64 (2) */
    int32_t shared_format; /* shared expert: MOE_FORMAT_INT4 (0), MOE_FORMAT_INT8 (1) or MOE_FORMAT_G64 (2) */
    int32_t ep_size;       /* expert parallelism: ranks sharing the layer's experts (0 or 1: none) */
    int32_t ep_rank;       /* this handle's rank, 0..ep_size-1 (see "Expert parallelism" below) */
} moe_config;

/* Expert parallelism (the reader.mx page, section 13, "五级专家驻留": disjoint
 * expert sets on the GPUs of one tier).  With ep_size = W > 1, rank r owns the
 * routed experts e with r*E/W <= e < (r+1)*E/W (integer division) and needs
 * only their slab and scale pointers (the others may be NULL); the shared
 * expert belongs to rank 0 (other ranks may pass NULL for it).  Every rank
 * runs the whole router (replicated router weights), so all ranks agree on the
 * selection, and moe_forward writes the rank's partial output
 *     y_r = sum over k with idx_k owned by r of w_k d_k
 *           (+ d_shared, and + x under MOE_FLAG_PRENORM_RESIDUAL, on rank 0 only);
 * the layer's y is the sum of y_r over the ranks: one all-reduce (or
 * reduce-scatter) of y[T, H], which the caller runs (e.g. NCCL, summing in a
 * fixed rank order).  EP handles take the generic kernels at every T (not the
 * single-kernel decode path). */

/* Weight formats of an expert slab:
 * INT4: gate [I, H/2] | up [I, H/2] | down [H, I/2] bytes, two values per byte
 *       (q + 8, low nibble first); scale buffer: one float32 per output row,
 *       sg [I] | su [I] | sd [H].
 * INT8: gate [I, H] | up [I, H] | down [H, I] bytes, one signed value per byte
 *       (the OLMoE engine of the reader.mx page, section 03); scales as INT4.
 * G64:  int4 affine, group size 64 (Edge0 article, section 三): the INT4 slab
 *       layout holding unsigned nibbles u in [0, 15]; the scale buffer holds one
 *       float16 pair (s, b) (s in the low half of each 4-byte word) per 64
 *       consecutive inputs of every row, gate [I][H/64] | up [I][H/64] |
 *       down [H][I/64], and W = s * u + b.
 * A config with an INT8 or G64 expert runs every call on the tensor-core expert
 * kernels and needs H, I and I_shared to be multiples of 128 (else
 * MOE_ERR_UNSUPPORTED); G64 weights are formed in f16 there (one rounding). */
#define MOE_FORMAT_INT4 0
#define MOE_FORMAT_INT8 1
#define MOE_FORMAT_G64 2

#define MOE_SCORE_SIGMOID 0   /* sigma = sigmoid(logit), selection by sigma + bias */
#define MOE_SCORE_SOFTMAX 1   /* g = softmax(logits), selection by g, bias unused */

/*
 * Weights are BORROWED device pointers: the caller allocates them, keeps them
 * alive and unchanged until moe_destroy, and frees them afterwards.  The two
 * per-expert pointer arrays themselves are HOST arrays of E entries; they are
 * copied at moe_init and not referenced afterwards.
 *
 * Expert slab (one per routed expert, and one for the shared expert), in the
 * expert's format (MOE_FORMAT_*, below); int4:
 *     gate q4 [I, H/2] | up q4 [I, H/2] | down q4 [H, I/2]     uint8, row-major
 * Expert scales:
 *     gate s [I] | up s [I] | down s [H]                        float32
 * Every slab and scale pointer must be 16-byte aligned.
 */
typedef struct moe_weights {
    const float *router_w;                  /* [E, H] float32, row-major */
    const float *router_bias;               /* [E] float32 (selection only) */
    const uint8_t *const *expert_slab;      /* host array of E device pointers */
    const float *const *expert_scale;       /* host array of E device pointers */
    const uint8_t *shared_slab;             /* NULL when n_shared == 0 */
    const float *shared_scale;              /* NULL when n_shared == 0 */
} moe_weights;

typedef struct moe_handle moe_handle;

/* Validates cfg and weights, allocates the handle's device workspace (sized
 * for max_tokens tokens per call) on the current device, and returns the
 * handle in *out.  On error *out is NULL and nothing stays allocated.  With
 * int4 experts and max_tokens >= 256 it also encodes a tensor-copy map of
 * every expert slab (the batched tensor-core path reads the weights through
 * them), so the weight buffers must stay where they are while the handle
 * lives, as for every other borrowed pointer. */
moe_status moe_init(const moe_config *cfg, const moe_weights *w, int32_t max_tokens,
                    moe_handle **out);

/* y[T,H] = step(x[T,H]); x and y are device float32, row-major, must not
 * overlap, and y is overwritten.  0 <= T <= max_tokens (T == 0 does nothing).
 * Launches on `stream` (a cudaStream_t; NULL = legacy default stream) and
 * returns without waiting.  Calls on one handle must not overlap on the GPU:
 * they share the handle's workspace.  The call may be captured in a CUDA
 * graph (stream capture): it keeps no per-call state on the host (the
 * single-kernel decode path counts its calls in device memory), so every
 * replay of a captured call computes the step on the x buffer's contents at
 * that time.  Not for capture: moe_forward_host (it synchronises) and calls
 * while moe_profile_start is recording. */
moe_status moe_forward(moe_handle *h, const float *x, int32_t T, float *y, void *stream);

/* As moe_forward, and also writes the router's choice: topk_idx[T,K] int32
 * (descending selection score), topk_w[T,K] float32, and, when not NULL,
 * expert_counts[E] int32 = tokens routed to each expert.  Device pointers. */
moe_status moe_forward_debug(moe_handle *h, const float *x, int32_t T, float *y,
                             int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                             void *stream);

/* Host-memory variant: copies x_host[T,H] to the device, runs the step on
 * `stream`, copies y back to y_host[T,H] and waits for the stream.  Host
 * buffers may be pageable; pinned buffers make the copies asynchronous. */
moe_status moe_forward_host(moe_handle *h, const float *x_host, int32_t T, float *y_host,
                            void *stream);

/* Frees the workspace and the handle (waits for the device first).  NULL is a no-op. */
moe_status moe_destroy(moe_handle *h);

/*
 * Per-kernel timing.  moe_profile_start(h, n) makes the next n forward calls
 * on h record a CUDA event on their stream before the first kernel and after
 * each kernel (n <= 4096; n == 0 stops recording and frees the events).
 * moe_profile_read waits for those events and returns, for each stage s,
 * stage_ms[s] = mean time from the event before stage s to the event after
 * it over the recorded calls.  Stages: 0 router (+ top-k, buckets),
 * 1 gate/up + SwiGLU, 2 down (+ combine for T == 1), 3 combine (T > 1 only;
 * 0 otherwise).  *n_calls = calls recorded.  stage_ms has MOE_PROFILE_STAGES
 * entries.
 */
#define MOE_PROFILE_STAGES 4
moe_status moe_profile_start(moe_handle *h, int32_t max_calls);
moe_status moe_profile_read(moe_handle *h, int32_t *n_calls, float *stage_ms);

/* Waits for the device, then reads and clears the handle's device error
 * word.  Kernels never wait without bound: a wait that runs out (a pipeline
 * stage, or a grid-wide barrier of the T == 1 kernel) sets a flag bit and the
 * kernel returns early.  That call's output is invalid, and so is the output of
 * every later call on the handle until this function has reset the handle's
 * barrier and call counters.  *flags = the bits seen (0: none); returns
 * MOE_ERR_CUDA when any was set, after that reset, so that later calls are
 * valid again. */
moe_status moe_device_error(moe_handle *h, uint32_t *flags);

/* Diagnosis and testing of the bounded waits (not a step of the method).
 * Moves the handle's device call counter ahead of its grid-barrier counters,
 * so that the next T == 1 call on the single-kernel decode path finds its first
 * grid barrier unreachable: that call's waits run out (after about 0.5 s), it
 * sets the device error word and returns without writing y.  moe_device_error
 * then reports the flag and resets the counters.  Waits for the device first.
 * MOE_ERR_UNSUPPORTED if T == 1 calls on the handle do not use that kernel. */
moe_status moe_debug_stall_next_call(moe_handle *h);

/* Testing of MOE_FLAG_DEBUG_CHECKS (not steps of the method).
 * moe_debug_check runs the checking kernel on `stream` over the routing and
 * buckets the handle's last call of T tokens left in its workspace (the
 * handle's flag is not needed); a failure sets MOE_DEVICE_ERR_CHECK and
 * *first_pair (after moe_device_error's wait: read it with moe_device_error)
 * -- see moe_debug_check_result.  moe_debug_set_topk overwrites one top-K
 * index of the workspace (pair = t * K + k, 0 <= pair < max_tokens * K) with
 * `expert` (any value: the checking kernel never uses an index it has not
 * checked), so that a test can make a check fail without running a step on
 * bad data.  Both wait for the device; MOE_ERR_INVALID on bad arguments. */
moe_status moe_debug_check(moe_handle *h, int32_t T);
moe_status moe_debug_set_topk(moe_handle *h, int32_t pair, int32_t expert);
/* After a failed check: *pair = a failing pair (t * K + k; or P + e for an
 * expert e's count, P = T * K), *code = which check (1 index range, 2 weight,
 * 3 repeated index, 4 position of another rank's pair, 5 position, 6 count or
 * offset, 7 owned-pair total); 0 / -1 when no check failed.  Call it before
 * moe_device_error (which clears the record). */
moe_status moe_debug_check_result(moe_handle *h, int32_t *pair, int32_t *code);

/* 1 if T == 1 calls on this handle run the single persistent decode kernel
 * (one block per SM, all of them resident together, meeting at grid-wide
 * barriers; weights streamed from HBM into registers; fixed-point activations
 * and dp4a), 0 if they use the generic kernels (shapes outside its limits: H,
 * I multiples of 32, I == I_shared, I <= 2048, H <= 8192, E <= 1024,
 * K + n_shared <= 32; the routing variants: n_group > 1 or the softmax score;
 * int8 or group-64 weights).  The kernel is launched so that it may start
 * while the previous kernel on the stream ends (programmatic dependent launch:
 * it reads only weights and pointer tables before that kernel is complete).
 * It needs every SM: while other work holds SMs, its barrier waits can run
 * out, which moe_device_error then reports. */
int32_t moe_uses_streaming_decode(const moe_handle *h);

/* Calls of up to this many tokens on h run one single-kernel decode step per
 * token, one after another on the stream (each step streams only its own
 * experts; below this size that is faster than the batched kernels, whose
 * per-call work is too small to keep the tensor cores fed).  0 when h does
 * not use the single-kernel decode path.  moe_forward_debug with
 * expert_counts always takes the batched kernels for T > 1. */
int32_t moe_streaming_decode_max_tokens(const moe_handle *h);

/* 1 if T > 1 calls on this handle run the experts on the tensor cores
 * (exact int4 weights times f16 activations, f32 accumulation: tcgen05.mma
 * with tensor-memory accumulators for T >= 256 with int4 experts, mma.sync
 * m16n8k16 otherwise), 0 if they use the CUDA-core batched kernels (exact f32
 * arithmetic; shapes where H, I or I_shared is not a multiple of 128, or
 * max_tokens == 1).  NULL -> 0. */
int32_t moe_uses_tensor_cores(const moe_handle *h);

/*
 * Timeline of the last T == 1 call on a handle created with MOE_FLAG_TRACE
 * (decode kernel only; a diagnostic of this library, not a step of the
 * method).  Waits for the device, then copies to out[b * MOE_TRACE_SLOTS + i]
 * (host memory, capacity_blocks * MOE_TRACE_SLOTS uint64 values) the GPU
 * global-timer readings, in nanoseconds, that block b of the decode launch
 * took at:
 *   0 its start            1 router scores and x digits written
 *   2 routing known        3 past the SwiGLU barrier
 *   4 its slots' h digits  5 past the down barrier      6 its end
 *   7 past the router-score barrier
 *   8 + i  warp 0 finished its i-th gate/up unit (i < 32)
 *   40 + i warp 0 finished its i-th down unit (i < 24)
 * Unreached entries are 0.  *n_blocks = blocks of the launch (copied:
 * min(*n_blocks, capacity_blocks)).  MOE_ERR_UNSUPPORTED if the handle was
 * created without MOE_FLAG_TRACE or does not use the decode kernel.
 */
#define MOE_TRACE_SLOTS 64
moe_status moe_trace_read(moe_handle *h, uint64_t *out, int32_t capacity_blocks, int32_t *n_blocks);

/* Device workspace moe_init would allocate for this config (0 if invalid). */
size_t moe_workspace_bytes(const moe_config *cfg, int32_t max_tokens);

/* Message of the last failure on this thread ("" if none). */
const char *moe_last_error(void);

int32_t moe_abi_version(void);

/*
 * Router only, with no device allocation.  (The pages have no counterpart:
 * this is a convenience of this library.)
 *
 * Some callers may not allocate device memory: a host framework whose device
 * memory all belongs to its own pool allocator, or a serving loop that must
 * not call cudaMalloc/cudaFree because those calls can synchronise the device
 * and can fail under memory pressure.  They cannot create a moe_handle, whose
 * moe_init allocates a workspace.  This call computes, for T tokens x[T,H]
 * (device float32), exactly what moe_forward_debug returns in topk_idx[T,K]
 * (int32, descending selection score) and topk_w[T,K] (float32): router
 * logits W_r x (with 1/rms(x) applied when cfg->flags has
 * MOE_FLAG_PRENORM_RESIDUAL), then the selection cfg describes: the sigmoid
 * family (top-K of sigmoid + bias, group-limited when n_group > 1) or the
 * softmax family (score_func = MOE_SCORE_SOFTMAX), each with or without
 * renormalisation (norm_topk) and times routed_scale, as described at the
 * top of this file.  The fields read are hidden, n_experts, top_k, n_group,
 * topk_group, score_func, norm_topk, routed_scale, rms_eps and flags; the
 * expert sizes and formats are ignored.
 *
 * Scratch: one fixed static device array in the library (logits of up to
 * MOE_ROUTE_NOALLOC_MAX_TOKENS x MOE_ROUTE_NOALLOC_MAX_EXPERTS floats plus a
 * ticket counter, about 32 KB), held by every GPU that loads the library
 * until the process exits.  The caller passes all inputs and outputs; the
 * call allocates nothing (no cudaMalloc, no cudaFree).  The first call on a
 * device looks the array's device address up with that device current (and
 * sets the kernel's shared-memory limit); make that first call before any
 * stream capture.  Every call shares the array: calls that overlap on the GPU
 * (other streams, other host threads on the same device) race and must be
 * serialised by the caller.  The call clears the ticket counter on `stream`
 * before its kernel; logits are rewritten in full every call.
 *
 * Errors: MOE_ERR_INVALID for NULL or misaligned pointers (router_w and x
 * 16-byte aligned), T outside 0..MOE_ROUTE_NOALLOC_MAX_TOKENS, and selection
 * fields that moe_init would also reject: top_k outside 1..min(n_experts, 32),
 * score_func not MOE_SCORE_SIGMOID or MOE_SCORE_SOFTMAX, n_group outside 1..32
 * or not dividing n_experts, n_group > 1 with the softmax score, topk_group
 * outside 1..n_group or top_k above topk_group * n_experts / n_group (when
 * n_group > 1), norm_topk not 0 or 1.  MOE_ERR_UNSUPPORTED for hidden not a
 * multiple of 32 in [32, 16384] or n_experts outside
 * 1..MOE_ROUTE_NOALLOC_MAX_EXPERTS.  MOE_ERR_CUDA if a CUDA call fails.
 * T == 0 does nothing.  This call does not set moe_last_error's message.
 */
#define MOE_ROUTE_NOALLOC_MAX_TOKENS 8
#define MOE_ROUTE_NOALLOC_MAX_EXPERTS 1024
moe_status moe_route_noalloc(const moe_config *cfg, const float *router_w, const float *router_bias,
                             const float *x, int32_t T, int32_t *topk_idx, float *topk_w,
                             void *stream);

#ifdef __cplusplus
}
#endif
#endif
