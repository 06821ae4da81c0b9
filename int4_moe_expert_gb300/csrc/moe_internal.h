// Internal declarations shared by the C-ABI layer (moe_abi.cu) and the
// kernels (moe_kernels.cu).  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Problem constants of one handle (validated by moe_init).
struct Dims {
    int H, E, K, I, n_shared, I_sh;
    int I_max;          // max(I, I_sh)
    int norm_topk;
    int n_group, topk_group;   // group-limited selection when n_group > 1
    int score_func;     // MOE_SCORE_SIGMOID / MOE_SCORE_SOFTMAX
    int expert_fmt, shared_fmt;   // MOE_FORMAT_INT4 / MOE_FORMAT_INT8
    int mma_fmt;        // an int8 or group-64 expert: every T runs the tensor-core expert kernels
    int tc;             // int4 experts: calls with T >= kTcMinT run them on tcgen05
    int prenorm;        // MOE_FLAG_PRENORM_RESIDUAL
    float scale;        // routed_scale
    float eps;          // rms_eps
    int max_tokens;
    int fast_decode;    // T == 1 runs the streaming kernels (moe_decode.cu)
    int mma;            // T > 1 runs the tensor-core expert kernels (H, I, I_sh multiples of 128)
    int trace;          // MOE_FLAG_TRACE: the decode kernel records its timeline
    int dec_grid;       // blocks of the decode launch (the GPU's SM count; 0 before prepare)
    int ep_lo, ep_hi;   // routed experts this handle computes: [ep_lo, ep_hi) ([0, E) without expert parallelism)
    int resid;          // add x to the output (pre-norm residual; rank 0 only under expert parallelism)
    int debug_checks;   // MOE_FLAG_DEBUG_CHECKS: a checking kernel after every call
};

// Device workspace owned by a handle.  Vectors marked "perm" are stored in
// the chunk-permuted order described in moe_kernels.cu (perm_pos).
struct Workspace {
    float *rnorm;        // [maxT] 1/rms(x_t) (1 when no pre-norm)
    float *xperm;        // [maxT, H] perm, x_t * rnorm_t
    float *logits;       // [maxT, E] raw router logits
    int *topk_idx;       // [maxT, K]
    float *topk_w;       // [maxT, K]
    unsigned *counters;  // [16] last-block tickets, reset by the last block
    float *h;            // [(maxT*K + maxT), I_max] perm, SwiGLU activations
    int *cnt;            // [E]
    int *off;            // [E+1]
    int *perm;           // [maxT*K] pair ids (t*K+k) grouped by expert, stable
    int *inv;            // [maxT*K] position of pair p in perm
    int *slot_expert;    // [E] active experts, ascending id
    int *n_slots;        // [1]
    float *dbuf;         // [(maxT*K + maxT), H] unweighted down outputs (T > 1)
    // T > 1 tensor-core path: f16 activations in mma order (mma_pos in moe_kernels.cu)
    uint16_t *x16;       // [maxT, H] pre-normed x
    uint16_t *h16;       // [(maxT*K + maxT), I_max] SwiGLU activations, rows as h (tcgen05 path:
                         //   the item-blocked layout of moe_kernels.cu, tc_act_index)
    uint16_t *xp16;      // tcgen05 gate/up: every work item's x16 rows in that layout (permute_x16_kernel)
    int tc_items;        // work items the tcgen05 layouts hold (0 without that path)
    int *items;          // [2 * max_items] (slot, first token) of every work item (item_tok tokens)
    int *n_items;        // [1]
    float *lpart;        // [S, T, E] tiled router: logits of each of a call's S k-ranges
    float *sspart;       // [S, T] tiled router: sums of squares of each k-range
    // decode (T == 1) single-kernel path (moe_decode.cu)
    unsigned *err;       // [4] device error word: bounded waits that ran out
    float *dpart;        // [kMaxSlots, H] down outputs per slot (times the routing weight)
    float *dscore;       // [2, E] decode router: sigmoid | selection score (sigmoid + bias)
    unsigned long long *trace;   // [kTraceBlocks, MOE_TRACE_SLOTS] decode timeline (MOE_FLAG_TRACE)
    size_t total_bytes;  // size of the carved region
};

constexpr int kMaxSlots = 33;   // K <= 32 routed + 1 shared
constexpr int kRouterMaxSplit = 32;  // tiled router: k-ranges (split-K) at most
constexpr int kItemTokens = 16;  // tokens of the smallest mma.sync work item (2 n8 tiles)
inline int max_items(int T, int K, int E, int n_shared, int item = kItemTokens) {   // work items, at most
    const int P = T * K;
    return P / item + (E < P ? E : P) + (n_shared ? (T + item - 1) / item : 0) + 1;
}
bool mma_supported(const Dims &d);
bool tc_supported(const Dims &d);   // int4 experts on the tensor-core path: tcgen05 for large T
// tcgen05 path (T >= its minimum): tensor maps of every expert's weights, kTmapBytes each,
// encoded once by moe_init: [2e] gate/up rows and [2e + 1] down rows of routed expert e
// ([2E], [2E + 1]: the shared expert)
constexpr int kTmapBytes = 128;
bool tc_maps_needed(const Dims &d);
size_t tc_map_count(const Dims &d);
struct Params;
// host_slabs: the routed experts' slab pointers (NULL: another rank's expert, no map)
cudaError_t upload_tc_maps(const Params &p, const uint8_t *const *host_slabs, void *dev);
constexpr int kTraceBlocks = 1024;   // decode blocks the trace buffer holds

// Everything a kernel needs, passed by value.
struct Params {
    Dims d;
    const float *router_w;
    const float *router_b;
    const uint8_t *const *slabs;    // device array [E]
    const float *const *scales;     // device array [E]
    const uint8_t *sh_slab;
    const float *sh_scale;
    Workspace ws;
    int item_tok;                   // this call: tokens per tensor-core work item
    const void *tmaps;              // tcgen05 path: device array of tensor maps (tc_map_count), else NULL
};

size_t workspace_bytes(const Dims &d);

// MOE_FLAG_DEBUG_CHECKS: the routing / bucket checks over the state of a call of T tokens
// (buckets: whether that call built them, buckets_built below).
cudaError_t launch_checks(const Params &p, int T, bool buckets, cudaStream_t st);
bool buckets_built(const Dims &d, int T, bool want_counts);
int decode_loop_max_tokens();   // calls of up to this many tokens run one decode step per token
void carve_workspace(const Dims &d, void *base, Workspace *ws);

// Per-config kernel attributes (dynamic shared memory limits); once per handle.
cudaError_t prepare_kernels(Dims &d);

constexpr int kStages = 4;   // router, gate/up, down, combine

// Decode path (moe_decode.cu): T == 1 as one persistent kernel (one block per SM, all resident).
// ws.counters[4..6] are its grid barriers: they only grow, by gridDim per
// call; ws.counters[7] counts the calls (read and advanced on the device, so
// the launch has no per-call host state and can be captured in a graph).
bool decode_fast_supported(const Dims &d);
cudaError_t prepare_decode_fast(Dims &d);   // sets d.dec_grid, or clears d.fast_decode for this GPU
int decode_grid_blocks(const Dims &d);      // blocks of the decode launch (0 before prepare)
cudaError_t launch_decode_fast(const Params &p, const float *x, float *y, cudaStream_t st, cudaEvent_t *ev,
                               bool want_counts);

// Launch the whole step for T >= 1 tokens on `stream`.  want_buckets forces
// the token -> expert histogram (ws.cnt) even for T == 1.  When ev is not
// NULL, ev[0] is recorded before the first kernel and ev[s+1] after stage s
// (kStages + 1 events; stages a path does not run get back-to-back events).
// Returns the first launch error (cudaSuccess when all launches were issued).
cudaError_t launch_forward(const Params &p, const float *x, int T, float *y, cudaStream_t stream,
                           bool want_buckets, cudaEvent_t *ev);

}  // namespace moe
