// Kernels of the int4 routed-MoE FFN step (sm_103a).
//
// Step order (GLM-5.2 operator breakdown, devpress.csdn.net, "Step 6 (MoE)"
// 6a-6d; reader.mx "25GB 内存上运行 GLM 5.2 744B", section 11):
//   router    logits = W_r x, sigma, + bias, top-K, renormalised weights
//   buckets   (T > 1) tokens grouped per expert, each expert read once per
//             batch (the batch union of section 11)
//   gate/up   g = s_g (Q_g x), u = s_u (Q_u x), h = silu(g) * u
//   down      d = s_d (Q_d h), y = sum_k w_k d_k + d_shared
//
// Vectors that feed an int4 dot product (x and h) are kept in a
// "chunk-permuted" order so that one 16-byte weight load (32 int4 values)
// meets its 32 activations as eight float4 loads that are contiguous across
// the lanes of a warp; see perm_pos.
#include <cuda.h>           // CUtensorMap and its enums (the encoder is resolved at run time)
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Tokens up to which a call on a single-kernel-decode handle runs one step per token instead of the
// batched kernels (measured on the GLM-5.2 layer: see the design notes)
constexpr int kDecodeLoopMaxT = 6;
constexpr int kGemvMaxT = 8;       // router GEMV handles up to this many tokens
constexpr int kGemvAhead = 4;      // router GEMV: row steps (32 lanes x 16 bytes) loaded at once
constexpr int kRouterBlocks = 456;  // tiled router: aim for 3 blocks per SM (split-K over H)

// ---------------------------------------------------------------------------
// Layout helpers
// ---------------------------------------------------------------------------

// Position of element i of a length-L vector (L % 32 == 0) in chunk-permuted
// order.  Chunk c holds elements 32c..32c+31.  Within a chunk, the 16 packed
// bytes are four 32-bit words; word m holds elements 8m..8m+7, with element
// 8m+2b in the low nibble and 8m+2b+1 in the high nibble of byte b.  The
// permuted vector is an array of float4: float4 (k*C + c) for k = 2m holds
// the even elements 8m+{0,2,4,6} of chunk c and k = 2m+1 the odd ones
// 8m+{1,3,5,7}.
__host__ __device__ __forceinline__ int perm_pos(int i, int L) {
    const int C = L >> 5;
    const int c = i >> 5, j = i & 31, m = j >> 3, e = j & 7;
    const int k = 2 * m + (e & 1), r = e >> 1;
    return ((k * C + c) << 2) + r;
}

// Position of element i of a vector in the f16 "mma order" of the T > 1
// tensor-core kernels: within each group of 8 consecutive elements the order
// is 0 4 1 5 2 6 3 7, so that one 32-bit word of packed int4 weights (8
// values) and the matching 16 bytes of activations split into the same four
// (element, element + 4) pairs; see mma_expert_kernel.
__host__ __device__ __forceinline__ int mma_pos(int i) {
    return (i & ~7) | ((i & 3) << 1) | ((i >> 2) & 1);
}

__device__ __forceinline__ uint16_t f2h_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }

// 16-byte streaming load of weights: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *ptr) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One int4 nibble (already isolated in byte b of v) to its exact float value
// q = nibble - 8: the byte becomes the low mantissa byte of 2^23 (0x4B000000),
// giving 2^23 + nibble exactly, then 2^23 + 8 is subtracted exactly.
__device__ __forceinline__ float nib(uint32_t v, uint32_t b) {
    return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440u | b)) - 8388616.0f;
}

// acc + sum over the 8 values of one packed word, against their activations:
// xe = elements 0,2,4,6 and xo = elements 1,3,5,7 of the word.
__device__ __forceinline__ float dot_word(uint32_t w, float4 xe, float4 xo, float acc) {
    const uint32_t lo = w & 0x0F0F0F0Fu;
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
    acc = fmaf(nib(lo, 0), xe.x, acc);
    acc = fmaf(nib(hi, 0), xo.x, acc);
    acc = fmaf(nib(lo, 1), xe.y, acc);
    acc = fmaf(nib(hi, 1), xo.y, acc);
    acc = fmaf(nib(lo, 2), xe.z, acc);
    acc = fmaf(nib(hi, 2), xo.z, acc);
    acc = fmaf(nib(lo, 3), xe.w, acc);
    acc = fmaf(nib(hi, 3), xo.w, acc);
    return acc;
}

// acc + dot(one 16-byte chunk of 32 int4 weights, its 32 permuted activations)
__device__ __forceinline__ float dot_chunk(uint4 w, const float4 (&xv)[8], float acc) {
    acc = dot_word(w.x, xv[0], xv[1], acc);
    acc = dot_word(w.y, xv[2], xv[3], acc);
    acc = dot_word(w.z, xv[4], xv[5], acc);
    acc = dot_word(w.w, xv[6], xv[7], acc);
    return acc;
}

__device__ __forceinline__ void load_chunk_act(const float *vec_perm, int C, int c, float4 (&xv)[8]) {
    const float4 *p4 = reinterpret_cast<const float4 *>(vec_perm);
#pragma unroll
    for (int k = 0; k < 8; k++) xv[k] = __ldg(p4 + k * C + c);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + expf(-g)) * u;
}

// ---------------------------------------------------------------------------
// Router: top-K selection and token -> expert buckets (last block of the
// router grid; no block ever waits on another)
// ---------------------------------------------------------------------------

// Order of the router's selection: larger score first, then lower index
// (the greedy strict-'>' scan of section 11 makes the lowest index win a tie).
__device__ __forceinline__ bool ranks_before(float v, int e, float bv, int be) {
    return v > bv || (v == bv && e < be);
}

// Top-K for tokens [t_begin, t_end): one warp per token.  Scores live in shared memory
// (sig and choice, E floats per warp).  NaN scores rank last, so an index in
// [0, E) is always produced.  Sigmoid family: sig = sigmoid(logit), choice =
// sig + bias, then (n_group > 1) the experts of all but the topk_group best
// groups are masked to -inf, a group's score being the sum of its two best
// choices.  Softmax family: sig = choice = softmax(logits).
__device__ void topk_phase(const Params &p, int t_begin, int t_end, float *smem) {
    const int E = p.d.E, K = p.d.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool softmax = p.d.score_func == MOE_SCORE_SOFTMAX;
    float *sig = smem + warp * 2 * E;
    float *choice = sig + E;
    for (int t = t_begin + warp; t < t_end; t += kWarps) {
        float lmax = -INFINITY;
        for (int base = 0; base < E; base += 256) {     // loads issued 8 at a time
            float lv[8], bv8[8];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int e = base + lane + 32 * i;
                lv[i] = e < E ? __ldcg(p.ws.logits + (size_t)t * E + e) : 0.0f;
                bv8[i] = e < E && !softmax ? p.router_b[e] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int e = base + lane + 32 * i;
                if (e < E) {
                    if (softmax) {
                        sig[e] = lv[i];
                        lmax = fmaxf(lmax, lv[i]);
                    } else {
                        const float s = 1.0f / (1.0f + expf(-lv[i]));
                        float c = s + bv8[i];
                        if (isnan(c)) c = -INFINITY;
                        sig[e] = s;
                        choice[e] = c;
                    }
                }
            }
        }
        if (softmax) {     // g = exp(l - max) / sum exp(l - max)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
            float z = 0.0f;
            for (int e = lane; e < E; e += 32) {
                const float v = expf(sig[e] - lmax);
                sig[e] = v;
                z += v;
            }
            z = warp_sum(z);
            for (int e = lane; e < E; e += 32) {
                const float g = sig[e] / z;
                sig[e] = g;
                choice[e] = isnan(g) ? -INFINITY : g;
            }
        }
        __syncwarp();
        if (p.d.n_group > 1) {
            // group `lane` (lane < n_group): the sum of its two best choices
            const int G = p.d.n_group, m = E / G;
            float gsc = -INFINITY;
            if (lane < G) {
                float b1 = -INFINITY, b2 = -INFINITY;
                for (int i = 0; i < m; i++) {
                    const float v = choice[lane * m + i];
                    if (v > b1) { b2 = b1; b1 = v; }
                    else if (v > b2) b2 = v;
                }
                gsc = m > 1 ? b1 + b2 : b1;
            }
            // keep the topk_group best groups (a tie goes to the lower group)
            uint32_t keep = 0u;
            bool taken = false;
            for (int r = 0; r < p.d.topk_group; r++) {
                float bv = taken ? -INFINITY : gsc;
                int be = (lane < G && !taken) ? lane : 0x7fffffff;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    if (ranks_before(ov, oe, bv, be)) { bv = ov; be = oe; }
                }
                keep |= 1u << be;
                if (lane == be) taken = true;
            }
            __syncwarp();
            for (int e = lane; e < E; e += 32)
                if (!((keep >> (e / m)) & 1u)) choice[e] = -INFINITY;
            __syncwarp();
        }
        uint32_t taken = 0;       // bit i: expert lane + 32 i already chosen
        float sum_sig = 0.0f, my_sig = 0.0f;
        int my_e = 0;
        for (int kk = 0; kk < K; kk++) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
            for (int i = 0; i * 32 + lane < E; i++) {
                if ((taken >> i) & 1u) continue;
                const int e = i * 32 + lane;
                const float v = choice[e];
                if (ranks_before(v, e, bv, be)) { bv = v; be = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ranks_before(ov, oe, bv, be)) { bv = ov; be = oe; }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            const float s = sig[be];
            sum_sig += s;               // same order in every lane
            if (lane == kk) { my_e = be; my_sig = s; }
        }
        // lane kk holds choice kk (K <= 32)
        if (lane < K) {
            const float den = softmax ? sum_sig : sum_sig + 1e-20f;
            p.ws.topk_idx[(size_t)t * K + lane] = my_e;
            p.ws.topk_w[(size_t)t * K + lane] = p.d.norm_topk ? p.d.scale * my_sig / den : p.d.scale * my_sig;
        }
        __syncwarp();
    }
}

__device__ void bucket_phase(const Params &p, int T, int *ismem) {
    const int E = p.d.E, K = p.d.K, P = T * K;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int *cnt = ismem;               // [E]
    int *run = cnt + E;             // [E] first position of each expert's pairs
    int *wcnt = run + E;            // [kWarps][E] pairs of each warp's range per expert, then
                                    // the warp's next position within the expert's pairs
    // warp w owns the pairs [q0, q1): its counts, then every warp's prefix per expert
    const int span = (P + kWarps - 1) / kWarps, q0 = min(P, warp * span), q1 = min(P, q0 + span);
    for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
    __syncthreads();
    for (int q = q0 + lane; q < q1; q += 32) {
        const int e = __ldcg(p.ws.topk_idx + q);
        if (e >= p.d.ep_lo && e < p.d.ep_hi) atomicAdd(&wcnt[warp * E + e], 1);   // expert parallelism: own experts only
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        int s = 0;
        for (int w = 0; w < kWarps; w++) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = s;
            s += c;
        }
        cnt[e] = s;
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scans of counts and of "active" flags, E <= 1024
        // (and of work items for the tensor-core kernels: p.item_tok tokens of one slot each)
        const int per = (E + 31) / 32;
        const int b = lane * per;
        const bool items = p.d.mma && (T > 1 || p.d.mma_fmt);
        int s = 0, a = 0, c = 0;
        for (int i = 0; i < per; i++) {
            const int e = b + i;
            if (e < E) { s += cnt[e]; a += cnt[e] > 0; c += (cnt[e] + p.item_tok - 1) / p.item_tok; }
        }
        int ps = s, pa = a, pc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vs = __shfl_up_sync(0xffffffffu, ps, o);
            const int va = __shfl_up_sync(0xffffffffu, pa, o);
            const int vc = __shfl_up_sync(0xffffffffu, pc, o);
            if (lane >= o) { ps += vs; pa += va; pc += vc; }
        }
        int off = ps - s, act = pa - a, it = pc - c;
        for (int i = 0; i < per; i++) {
            const int e = b + i;
            if (e < E) {
                p.ws.cnt[e] = cnt[e];
                p.ws.off[e] = off;
                run[e] = off;
                if (cnt[e] > 0) {
                    if (items)
                        for (int n0 = 0; n0 < cnt[e]; n0 += p.item_tok, it++) {
                            p.ws.items[2 * it] = act;
                            p.ws.items[2 * it + 1] = n0;
                        }
                    p.ws.slot_expert[act++] = e;
                }
                off += cnt[e];
            }
        }
        if (lane == 31) {
            p.ws.off[E] = ps;
            *p.ws.n_slots = pa;
            if (items) {                 // the shared expert: slot n_slots, all T tokens
                int n = pc;
                if (p.d.n_shared)
                    for (int n0 = 0; n0 < T; n0 += p.item_tok, n++) {
                        p.ws.items[2 * n] = pa;
                        p.ws.items[2 * n + 1] = n0;
                    }
                *p.ws.n_items = n;
            }
        }
    }
    __syncthreads();
    // each warp places its own pairs in order (pairs of one expert: warp ranges in order,
    // then q ascending within a range), 32 at a time
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = q0; base < q1; base += 32) {
        const int q = base + lane;
        int e = q < q1 ? __ldcg(p.ws.topk_idx + q) : -1;
        if (e >= 0 && (e < p.d.ep_lo || e >= p.d.ep_hi)) {   // another rank's expert: no position
            p.ws.inv[q] = -1;
            e = -1;
        }
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int lrank = __popc(same & lt_mask);
        if (e >= 0) {
            const int pos = run[e] + wcnt[warp * E + e] + lrank;
            p.ws.perm[pos] = q;
            p.ws.inv[q] = pos;
        }
        __syncwarp();
        if (e >= 0 && lrank == 0) wcnt[warp * E + e] += __popc(same);
        __syncwarp();
    }
}

// Shared tail of both router kernels: every block signs in; the last one to
// arrive sees all logits and runs top-K (and the buckets when asked).
__device__ void router_tail(const Params &p, int T, int buckets, unsigned nblocks, float *smem) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(p.ws.counters, 1u);
        s_last = (prev == nblocks - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    topk_phase(p, 0, T, smem);
    __syncthreads();
    if (buckets) bucket_phase(p, T, reinterpret_cast<int *>(smem));
    if (threadIdx.x == 0) *p.ws.counters = 0u;     // ready for the next call
}

// Router logits of experts 2 blockIdx.x and 2 blockIdx.x + 1 for T <= kGemvMaxT tokens,
// scaled by s_r[t]: warps 4 r .. 4 r + 3 share expert row r, each a quarter of H; the
// quarters' sums are added in order.  Every thread of the block calls it.
__device__ void gemv_logits(const Params &p, const float *__restrict__ x, int T, const float *s_r) {
    __shared__ float s_part[kWarps][kGemvMaxT];
    const int H = p.d.H, E = p.d.E, H4 = H / 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 2 + (warp >> 2), part = warp & 3;
    const int per = (H4 + 3) / 4, i0 = part * per, i1 = min(H4, i0 + per);
    float acc[kGemvMaxT];
#pragma unroll
    for (int t = 0; t < kGemvMaxT; t++) acc[t] = 0.0f;
    if (e < E) {
        const float4 *w4 = reinterpret_cast<const float4 *>(p.router_w + (size_t)e * H);
        int i = i0 + lane;
        // kGemvAhead steps of the row at once (their loads in flight together); the sums
        // still run in step order
        for (; i + 32 * (kGemvAhead - 1) < i1; i += 32 * kGemvAhead) {
            float4 wv[kGemvAhead];
#pragma unroll
            for (int u = 0; u < kGemvAhead; u++) wv[u] = __ldg(w4 + i + 32 * u);
#pragma unroll
            for (int t = 0; t < kGemvMaxT; t++) {
                if (t < T) {
                    float4 xv[kGemvAhead];
#pragma unroll
                    for (int u = 0; u < kGemvAhead; u++)
                        xv[u] = __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * H) + i + 32 * u);
#pragma unroll
                    for (int u = 0; u < kGemvAhead; u++) {
                        acc[t] = fmaf(wv[u].x, xv[u].x, acc[t]);
                        acc[t] = fmaf(wv[u].y, xv[u].y, acc[t]);
                        acc[t] = fmaf(wv[u].z, xv[u].z, acc[t]);
                        acc[t] = fmaf(wv[u].w, xv[u].w, acc[t]);
                    }
                }
            }
        }
        for (; i < i1; i += 32) {
            const float4 wv = __ldg(w4 + i);
#pragma unroll
            for (int t = 0; t < kGemvMaxT; t++) {
                if (t < T) {
                    const float4 xv = __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * H) + i);
                    acc[t] = fmaf(wv.x, xv.x, acc[t]);
                    acc[t] = fmaf(wv.y, xv.y, acc[t]);
                    acc[t] = fmaf(wv.z, xv.z, acc[t]);
                    acc[t] = fmaf(wv.w, xv.w, acc[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kGemvMaxT; t++) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) s_part[warp][t] = v;
    }
    __syncthreads();
    if (threadIdx.x < 2 * kGemvMaxT) {
        const int r = threadIdx.x / kGemvMaxT, t = threadIdx.x % kGemvMaxT, er = blockIdx.x * 2 + r;
        if (er < E && t < T) {
            const float v = s_part[4 * r][t] + s_part[4 * r + 1][t] + s_part[4 * r + 2][t] + s_part[4 * r + 3][t];
            p.ws.logits[(size_t)t * E + er] = v * s_r[t];
        }
    }
}

// Router for T <= kGemvMaxT tokens: four warps per expert row (gemv_logits).  Also writes
// rnorm and the permuted (and pre-normed) activations used by gate/up.
__global__ void __launch_bounds__(kThreads) router_gemv_kernel(Params p, const float *__restrict__ x,
                                                               int T, int buckets) {
    extern __shared__ float smem[];
    __shared__ float s_r[kGemvMaxT];
    const int H = p.d.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < T) {
        float ss = 0.0f;
        if (p.d.prenorm) {
            const float4 *x4 = reinterpret_cast<const float4 *>(x + (size_t)warp * H);
            for (int i = lane; i < H / 4; i += 32) {
                const float4 v = __ldg(x4 + i);
                ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
            }
            ss = warp_sum(ss);
        }
        const float r = p.d.prenorm ? 1.0f / sqrtf(ss / (float)H + p.d.eps) : 1.0f;
        if (lane == 0) {
            s_r[warp] = r;
            if (blockIdx.x == 0) p.ws.rnorm[warp] = r;
        }
    }
    __syncthreads();
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < T * H; i += gridDim.x * kThreads) {
        const int t = i / H, c = i - t * H;
        const float v = x[i] * s_r[t];
        p.ws.xperm[(size_t)t * H + perm_pos(c, H)] = v;
        if (p.d.mma && (T > 1 || p.d.mma_fmt)) p.ws.x16[(size_t)t * H + mma_pos(c)] = f2h_bits(v);
    }
    gemv_logits(p, x, T, s_r);
    router_tail(p, T, buckets, gridDim.x, smem);
}


// Router for T > kGemvMaxT tokens: the fp32 product logits[t][e] = sum_h x[t][h] W[e][h]
// (router GEMV of section 11, as a small GEMM) over 64-token x 64-expert tiles, the
// reduction split into gridDim.z k-ranges (whole 32-element stages).  Each stage of x
// and W rows goes through a kRtStages-slot cp.async ring (rows padded to kRtLd floats);
// thread (th, ty, tx) of warp 2 eq + th keeps a 4 x 4 block of sums, tokens
// 32 th + ty + 8 j and experts 16 eq + tx + 4 i, and reads float4s along k, so each
// shared-memory read serves 8 (tokens) or 4 (experts) lanes at once, conflict-free.
// Every block writes its k-range's partial logits (and, for pre-norm, the tokens'
// partial sums of squares); router_reduce_kernel adds them.  Deterministic: every sum
// has a fixed order.
constexpr int kRtTok = 64, kRtExp = 64, kRtK = 32, kRtStages = 4, kRtLd = kRtK + 4;
constexpr int kRtCv = 4;                               // activation steps a thread loads at once
constexpr size_t kRtSmem = (size_t)kRtStages * 2 * 64 * kRtLd * sizeof(float);

__device__ __forceinline__ void rt_cp16(uint32_t dst, const void *src, uint32_t bytes) {   // bytes 0: zero fill
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void rt_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void rt_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(kThreads) router_tiled_kernel(Params p, const float *__restrict__ x,
                                                                int T) {
    extern __shared__ __align__(16) float smem[];
    const int H = p.d.H, E = p.d.E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e0 = blockIdx.x * kRtExp, t0 = blockIdx.y * kRtTok;
    const int th = warp & 1, eq = warp >> 1, ty = lane >> 2, tx = lane & 3;
    const int nk = H / kRtK, z = blockIdx.z, S = gridDim.z;
    const int kb0 = (int)((long)z * nk / S), nkb = (int)((long)(z + 1) * nk / S) - kb0;
    const bool want_ss = p.d.prenorm && blockIdx.x == 0;    // block-uniform
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    // stage kb into its slot: 64 x rows then 64 W rows of 8 16-byte pieces, 4 pieces per thread
    auto issue = [&](int kb) {
        if (kb < nkb) {
            const int slot = kb % kRtStages;
            const int k0 = (kb0 + kb) * kRtK;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int c = tid + kThreads * (q & 1), row = c >> 3, piece = c & 7;
                const bool isw = q >= 2;
                const int g = (isw ? e0 : t0) + row;
                const bool ok = g < (isw ? E : T);
                const float *src = (isw ? p.router_w : x) + (size_t)(ok ? g : 0) * H + k0 + 4 * piece;
                const uint32_t dst = sbase + (uint32_t)((((2 * slot + (isw ? 1 : 0)) * 64 + row) * kRtLd + 4 * piece) * 4);
                rt_cp16(dst, src, ok ? 16u : 0u);
            }
        }
        rt_commit();
    };
    float acc[4][4], ss[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        ss[j] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; i++) acc[j][i] = 0.0f;
    }
#pragma unroll
    for (int k = 0; k < kRtStages - 1; k++) issue(k);
#pragma unroll 1
    for (int kb = 0; kb < nkb; kb++) {
        rt_wait<kRtStages - 2>();     // stage kb has landed (this thread's pieces)
        __syncthreads();              // ... everyone's; and everyone is done with stage kb - 1
        issue(kb + kRtStages - 1);    // into stage kb - 1's slot
        const float *X = smem + (size_t)(2 * (kb % kRtStages)) * 64 * kRtLd;
        const float *Wr = X + 64 * kRtLd;
#pragma unroll
        for (int k4 = 0; k4 < kRtK / 4; k4++) {
            float4 xa[4], wb[4];
#pragma unroll
            for (int j = 0; j < 4; j++) xa[j] = *reinterpret_cast<const float4 *>(X + (32 * th + ty + 8 * j) * kRtLd + 4 * k4);
#pragma unroll
            for (int i = 0; i < 4; i++) wb[i] = *reinterpret_cast<const float4 *>(Wr + (16 * eq + tx + 4 * i) * kRtLd + 4 * k4);
#pragma unroll
            for (int j = 0; j < 4; j++)
#pragma unroll
                for (int i = 0; i < 4; i++)
                    acc[j][i] = fmaf(xa[j].w, wb[i].w, fmaf(xa[j].z, wb[i].z, fmaf(xa[j].y, wb[i].y, fmaf(xa[j].x, wb[i].x, acc[j][i]))));
            if (want_ss) {
#pragma unroll
                for (int j = 0; j < 4; j++)
                    ss[j] = fmaf(xa[j].w, xa[j].w, fmaf(xa[j].z, xa[j].z, fmaf(xa[j].y, xa[j].y, fmaf(xa[j].x, xa[j].x, ss[j]))));
            }
        }
    }
    rt_wait<0>();
    // this k-range's partial logits [z][t][e] (and sums of squares [z][t])
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int t = t0 + 32 * th + ty + 8 * j;
        if (t < T) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int e = e0 + 16 * eq + tx + 4 * i;
                if (e < E) p.ws.lpart[((size_t)z * T + t) * E + e] = acc[j][i];
            }
            if (want_ss && eq == 0 && tx == 0) p.ws.sspart[(size_t)z * T + t] = ss[j];
        }
    }
}

// Second router kernel of a T > kGemvMaxT call, one block per token: the token's 1/rms
// (pre-norm), its logits = (sum of the k-range partials, in k-range order) / rms, its
// activations for the expert kernels (x / rms: f16 in mma order for the tensor-core path,
// f32 chunk-permuted for the CUDA-core path), then its top-K (warp 0); the last block to
// finish builds the buckets.  One block per token keeps every SM's share of the partial
// and activation traffic small.
__global__ void __launch_bounds__(kThreads) router_reduce_kernel(Params p, const float *__restrict__ x, int T,
                                                                 int S, int buckets) {
    extern __shared__ __align__(16) float smem[];
    __shared__ float s_red[kWarps];
    __shared__ int s_last;
    const int H = p.d.H, E = p.d.E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x;
    float r = 1.0f;
    if (p.d.prenorm) {
        float sq = 0.0f;
        if (warp == 0) {
            for (int k = lane; k < S; k += 32) sq += __ldcg(p.ws.sspart + (size_t)k * T + t);
            // the k-range order of the sum is fixed by the butterfly
            sq = warp_sum(sq);
            if (lane == 0) s_red[0] = sq;
        }
        __syncthreads();
        r = 1.0f / sqrtf(s_red[0] / (float)H + p.d.eps);
    }
    if (tid == 0) p.ws.rnorm[t] = r;
    for (int e = tid; e < E; e += kThreads) {
        float v = 0.0f;
        for (int k0 = 0; k0 < S; k0 += 16) {      // 16 partials in flight, added in k-range order
            float pv[16];
#pragma unroll
            for (int k = 0; k < 16; k++)
                pv[k] = k0 + k < S ? __ldcg(p.ws.lpart + ((size_t)(k0 + k) * T + t) * E + e) : 0.0f;
#pragma unroll
            for (int k = 0; k < 16; k++)
                if (k0 + k < S) v += pv[k];
        }
        p.ws.logits[(size_t)t * E + e] = v * r;
    }
    // activations, 8 elements per thread per step, kRtCv steps' loads in flight at once
    for (int c0 = 8 * tid; c0 < H; c0 += 8 * kThreads * kRtCv) {
        float4 va[kRtCv], vb[kRtCv];
#pragma unroll
        for (int u = 0; u < kRtCv; u++) {
            const int c = c0 + 8 * kThreads * u;
            if (c < H) {
                va[u] = __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * H + c));
                vb[u] = __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * H + c) + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < kRtCv; u++) {
            const int c = c0 + 8 * kThreads * u;
            if (c < H) {
                const float4 a = va[u], b = vb[u];
                const float v[8] = {a.x * r, a.y * r, a.z * r, a.w * r, b.x * r, b.y * r, b.z * r, b.w * r};
                if (p.d.mma) {       // group order 0 4 1 5 2 6 3 7
                    uint4 o;
                    o.x = (uint32_t)f2h_bits(v[0]) | ((uint32_t)f2h_bits(v[4]) << 16);
                    o.y = (uint32_t)f2h_bits(v[1]) | ((uint32_t)f2h_bits(v[5]) << 16);
                    o.z = (uint32_t)f2h_bits(v[2]) | ((uint32_t)f2h_bits(v[6]) << 16);
                    o.w = (uint32_t)f2h_bits(v[3]) | ((uint32_t)f2h_bits(v[7]) << 16);
                    *reinterpret_cast<uint4 *>(p.ws.x16 + (size_t)t * H + c) = o;
                } else {
#pragma unroll
                    for (int j = 0; j < 8; j++) p.ws.xperm[(size_t)t * H + perm_pos(c + j, H)] = v[j];
                }
            }
        }
    }
    __syncthreads();              // this token's logits are written
    topk_phase(p, t, t + 1, smem);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(p.ws.counters, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (buckets) bucket_phase(p, T, reinterpret_cast<int *>(smem));
    if (tid == 0) *p.ws.counters = 0u;
}

// ---------------------------------------------------------------------------
// Decode (T == 1): slot j < K is the j-th routed choice, slot K the shared expert
// ---------------------------------------------------------------------------

template <int RPW>
__global__ void __launch_bounds__(kThreads) gateup_decode_kernel(Params p) {
    const int H = p.d.H, C = H >> 5;
    const int slot = blockIdx.y;
    const uint8_t *slab;
    const float *sc;
    int Is;
    if (slot < p.d.K) {
        const int e = p.ws.topk_idx[slot];
        if (e < p.d.ep_lo || e >= p.d.ep_hi) return;   // another rank's expert (expert parallelism)
        slab = p.slabs[e];
        sc = p.scales[e];
        Is = p.d.I;
    } else {
        slab = p.sh_slab;
        sc = p.sh_scale;
        Is = p.d.I_sh;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kWarps + warp) * RPW;
    if (row0 >= Is) return;
    const size_t rb = (size_t)(H >> 1);
    const uint8_t *g0 = slab + (size_t)row0 * rb;
    const uint8_t *u0 = slab + ((size_t)Is + row0) * rb;
    float ag[RPW], au[RPW];
#pragma unroll
    for (int r = 0; r < RPW; r++) { ag[r] = 0.f; au[r] = 0.f; }
#pragma unroll 2
    for (int c = lane; c < C; c += 32) {
        uint4 wg[RPW], wu[RPW];
#pragma unroll
        for (int r = 0; r < RPW; r++) {
            wg[r] = ld_stream(g0 + r * rb + (size_t)c * 16);
            wu[r] = ld_stream(u0 + r * rb + (size_t)c * 16);
        }
        float4 xv[8];
        load_chunk_act(p.ws.xperm, C, c, xv);
#pragma unroll
        for (int r = 0; r < RPW; r++) {
            ag[r] = dot_chunk(wg[r], xv, ag[r]);
            au[r] = dot_chunk(wu[r], xv, au[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; r++) {
        const float g = warp_sum(ag[r]);
        const float u = warp_sum(au[r]);
        if (lane == r) {
            const int o = row0 + r;
            const float hv = silu_mul(sc[o] * g, sc[Is + o] * u);
            p.ws.h[(size_t)slot * p.d.I_max + perm_pos(o, Is)] = hv;
        }
    }
}


template <int RPW>
__global__ void __launch_bounds__(kThreads) down_decode_kernel(Params p, const float *__restrict__ x,
                                                               float *__restrict__ y) {
    __shared__ const uint8_t *s_slab[kMaxSlots];
    __shared__ const float *s_sc[kMaxSlots];
    __shared__ float s_w[kMaxSlots];
    const int H = p.d.H, K = p.d.K, I = p.d.I, Ish = p.d.I_sh;
    const int J = K + p.d.n_shared;
    if (threadIdx.x < J) {
        const int j = threadIdx.x;
        if (j < K) {
            const int e = p.ws.topk_idx[j];
            const bool own = e >= p.d.ep_lo && e < p.d.ep_hi;   // expert parallelism: own experts only
            s_slab[j] = own ? p.slabs[e] : nullptr;
            s_sc[j] = own ? p.scales[e] : nullptr;
            s_w[j] = p.ws.topk_w[j];
        } else {
            s_slab[j] = p.sh_slab;
            s_sc[j] = p.sh_scale;
            s_w[j] = 1.0f;
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kWarps + warp) * RPW;
    if (row0 >= H) return;
    const int C = I >> 5, Csh = Ish >> 5;
    const int Qr = K * C;
    const int Q = Qr + (p.d.n_shared ? Csh : 0);
    float acc[RPW];
#pragma unroll
    for (int r = 0; r < RPW; r++) acc[r] = 0.f;
    // (slot, chunk) items strided over the lanes; every item adds
    // w_j * s_d[o] * dot(Q_d[o, chunk], h_j[chunk]) to row o.
#pragma unroll 2
    for (int q = lane; q < Q; q += 32) {
        int j, c, Ij;
        if (q < Qr) { j = q / C; c = q - j * C; Ij = I; }
        else { j = K; c = q - Qr; Ij = Ish; }
        if (s_slab[j] == nullptr) continue;
        const size_t rbI = (size_t)(Ij >> 1);
        const uint8_t *d0 = s_slab[j] + 2 * (size_t)Ij * (size_t)(H >> 1) + (size_t)row0 * rbI + (size_t)c * 16;
        uint4 wv[RPW];
#pragma unroll
        for (int r = 0; r < RPW; r++) wv[r] = ld_stream(d0 + r * rbI);
        float4 hv[8];
        load_chunk_act(p.ws.h + (size_t)j * p.d.I_max, Ij >> 5, c, hv);
        const float *sd = s_sc[j] + 2 * Ij;
        const float wj = s_w[j];
#pragma unroll
        for (int r = 0; r < RPW; r++) {
            const float part = dot_chunk(wv[r], hv, 0.0f);
            acc[r] = fmaf(wj * sd[row0 + r], part, acc[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; r++) {
        const float v = warp_sum(acc[r]);
        if (lane == r) {
            const int o = row0 + r;
            y[o] = p.d.resid ? x[o] + v : v;
        }
    }
}

// ---------------------------------------------------------------------------
// Batched (T > 1): slot s < n_slots is the s-th active expert with its tokens,
// slot n_slots the shared expert over all T tokens.
// ---------------------------------------------------------------------------

struct SlotInfo {
    const uint8_t *slab;
    const float *sc;
    int Is;          // intermediate size of this expert
    int n;           // tokens in the slot
    int base;        // first position in perm (routed) or -1 (shared)
    bool valid;
};

__device__ __forceinline__ SlotInfo slot_info(const Params &p, int T, int slot) {
    SlotInfo s;
    const int ns = *p.ws.n_slots;
    s.valid = true;
    if (slot < ns) {
        const int e = p.ws.slot_expert[slot];
        s.slab = p.slabs[e];
        s.sc = p.scales[e];
        s.Is = p.d.I;
        s.n = p.ws.cnt[e];
        s.base = p.ws.off[e];
    } else if (slot == ns && p.d.n_shared) {
        s.slab = p.sh_slab;
        s.sc = p.sh_scale;
        s.Is = p.d.I_sh;
        s.n = T;
        s.base = -1;
    } else {
        s.valid = false;
        s.slab = nullptr; s.sc = nullptr; s.Is = 0; s.n = 0; s.base = 0;
    }
    return s;
}

// token index and h/d row of the u-th token of a slot
__device__ __forceinline__ void slot_token(const Params &p, const SlotInfo &s, int T, int u,
                                           int *tok, int *row) {
    if (s.base < 0) { *tok = u; *row = T * p.d.K + u; }
    else { const int pos = s.base + u; *tok = p.ws.perm[pos] / p.d.K; *row = pos; }
}

template <int RPW, int NT>
__global__ void __launch_bounds__(kThreads) gateup_batched_kernel(Params p, int T) {
    const SlotInfo s = slot_info(p, T, blockIdx.y);
    if (!s.valid) return;
    const int H = p.d.H, C = H >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kWarps + warp) * RPW;
    if (row0 >= s.Is) return;
    const size_t rb = (size_t)(H >> 1);
    const uint8_t *g0 = s.slab + (size_t)row0 * rb;
    const uint8_t *u0 = s.slab + ((size_t)s.Is + row0) * rb;
    for (int tb = 0; tb < s.n; tb += NT) {
        int tok[NT], hrow[NT];
#pragma unroll
        for (int u = 0; u < NT; u++) {
            if (tb + u < s.n) slot_token(p, s, T, tb + u, &tok[u], &hrow[u]);
            else { tok[u] = 0; hrow[u] = -1; }
        }
        float ag[NT][RPW], au[NT][RPW];
#pragma unroll
        for (int u = 0; u < NT; u++)
#pragma unroll
            for (int r = 0; r < RPW; r++) { ag[u][r] = 0.f; au[u][r] = 0.f; }
        for (int c = lane; c < C; c += 32) {
            uint4 wg[RPW], wu[RPW];
#pragma unroll
            for (int r = 0; r < RPW; r++) {
                wg[r] = ld_stream(g0 + r * rb + (size_t)c * 16);
                wu[r] = ld_stream(u0 + r * rb + (size_t)c * 16);
            }
#pragma unroll
            for (int u = 0; u < NT; u++) {
                if (hrow[u] < 0) continue;
                float4 xv[8];
                load_chunk_act(p.ws.xperm + (size_t)tok[u] * H, C, c, xv);
#pragma unroll
                for (int r = 0; r < RPW; r++) {
                    ag[u][r] = dot_chunk(wg[r], xv, ag[u][r]);
                    au[u][r] = dot_chunk(wu[r], xv, au[u][r]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < NT; u++) {
#pragma unroll
            for (int r = 0; r < RPW; r++) {
                const float g = warp_sum(ag[u][r]);
                const float uu = warp_sum(au[u][r]);
                if (lane == r && hrow[u] >= 0) {
                    const int o = row0 + r;
                    p.ws.h[(size_t)hrow[u] * p.d.I_max + perm_pos(o, s.Is)] =
                        silu_mul(s.sc[o] * g, s.sc[s.Is + o] * uu);
                }
            }
        }
    }
}

template <int RPW, int NT>
__global__ void __launch_bounds__(kThreads) down_batched_kernel(Params p, int T) {
    const SlotInfo s = slot_info(p, T, blockIdx.y);
    if (!s.valid) return;
    const int H = p.d.H, Cj = s.Is >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kWarps + warp) * RPW;
    if (row0 >= H) return;
    const size_t rbI = (size_t)(s.Is >> 1);
    const uint8_t *d0 = s.slab + 2 * (size_t)s.Is * (size_t)(H >> 1) + (size_t)row0 * rbI;
    const float *sd = s.sc + 2 * s.Is;
    for (int tb = 0; tb < s.n; tb += NT) {
        int tok[NT], hrow[NT];
#pragma unroll
        for (int u = 0; u < NT; u++) {
            if (tb + u < s.n) slot_token(p, s, T, tb + u, &tok[u], &hrow[u]);
            else { tok[u] = 0; hrow[u] = -1; }
        }
        float acc[NT][RPW];
#pragma unroll
        for (int u = 0; u < NT; u++)
#pragma unroll
            for (int r = 0; r < RPW; r++) acc[u][r] = 0.f;
        for (int c = lane; c < Cj; c += 32) {
            uint4 wv[RPW];
#pragma unroll
            for (int r = 0; r < RPW; r++) wv[r] = ld_stream(d0 + r * rbI + (size_t)c * 16);
#pragma unroll
            for (int u = 0; u < NT; u++) {
                if (hrow[u] < 0) continue;
                float4 hv[8];
                load_chunk_act(p.ws.h + (size_t)hrow[u] * p.d.I_max, Cj, c, hv);
#pragma unroll
                for (int r = 0; r < RPW; r++) acc[u][r] = dot_chunk(wv[r], hv, acc[u][r]);
            }
        }
#pragma unroll
        for (int u = 0; u < NT; u++) {
#pragma unroll
            for (int r = 0; r < RPW; r++) {
                const float v = warp_sum(acc[u][r]);
                if (lane == r && hrow[u] >= 0) {
                    const int o = row0 + r;
                    p.ws.dbuf[(size_t)hrow[u] * H + o] = sd[o] * v;
                }
            }
        }
    }
}

// y[t] = sum_k w[t,k] d[(t,k)] (k ascending) + d_shared[t] (+ x[t] with pre-norm residual)
// Grid (T, ceil(H / (4 kThreads))): four consecutive outputs per thread.
__global__ void __launch_bounds__(kThreads) combine_kernel(Params p, const float *__restrict__ x,
                                                           float *__restrict__ y, int T) {
    const int t = blockIdx.x, H = p.d.H, K = p.d.K;
    const int o = (blockIdx.y * kThreads + threadIdx.x) * 4;
    if (o >= H) return;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; k++) {
        const int q = t * K + k;
        const int pos = p.ws.inv[q];
        if (pos < 0) continue;          // another rank's expert (expert parallelism)
        const float w = p.ws.topk_w[q];
        const float4 d = __ldg(reinterpret_cast<const float4 *>(p.ws.dbuf + (size_t)pos * H + o));
        v.x = fmaf(w, d.x, v.x);
        v.y = fmaf(w, d.y, v.y);
        v.z = fmaf(w, d.z, v.z);
        v.w = fmaf(w, d.w, v.w);
    }
    if (p.d.n_shared) {
        const float4 d = __ldg(reinterpret_cast<const float4 *>(p.ws.dbuf + (size_t)(T * K + t) * H + o));
        v.x += d.x; v.y += d.y; v.z += d.z; v.w += d.w;
    }
    if (p.d.resid) {
        const float4 r = __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * H + o));
        v.x += r.x; v.y += r.y; v.z += r.z; v.w += r.w;
    }
    *reinterpret_cast<float4 *>(y + (size_t)t * H + o) = v;
}

// ---------------------------------------------------------------------------
// Batched (T > 1) on the tensor cores: mma.sync m16n8k16, f16 x f16 -> f32.
//
// A = int4 weight rows (exact in f16), B = f16 activations of up to
// 16 or 32 tokens (one work item: a slot and a run of its tokens), C in
// f32 registers.  Each thread streams, per 128-element block of the reduction,
// the 16 bytes at offset 16 q (q = lane % 4) of each of its weight rows: four
// 32-bit words of 8 int4 values.  One word w splits with two masks and two
// shifts into the f16 pairs (e0, e4), (e1, e5), (e2, e6), (e3, e7) (1024 + n
// or 1024 + 16 n in the f16 bit pattern, then one subtract or fma), and the
// mma order of the activations (mma_pos) stores each 8-element group as
// 0 4 1 5 2 6 3 7, so the same pairs are adjacent f16 values there.  Word w
// of thread q covers two k-steps: pairs (e0,e4) / (e1,e5) are the fragment's
// columns (2q, 2q+1) / (2q+8, 2q+9) of the first, (e2,e6) / (e3,e7) of the
// second.  A dot product does not depend on the order of its terms, so A and B
// only have to agree on it, which they do.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
// 8 packed int4 values (q + 8, element 2b in the low nibble of byte b) -> the
// f16x2 pairs (e0,e4), (e1,e5), (e2,e6), (e3,e7), exact.
__device__ __forceinline__ void int4x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    constexpr uint32_t kMagic = 0x64006400u;   // f16 1024 in both halves
    constexpr uint32_t kSubLo = 0x64086408u;   // 1032 = 1024 + 8
    constexpr uint32_t kMulHi = 0x2C002C00u;   // 1/16
    constexpr uint32_t kAddHi = 0xD480D480u;   // -72 = -(1024/16 + 8)
    h[0] = h2_sub((w & 0x000F000Fu) | kMagic, kSubLo);
    h[1] = h2_fma((w & 0x00F000F0u) | kMagic, kMulHi, kAddHi);
    h[2] = h2_sub(((w >> 8) & 0x000F000Fu) | kMagic, kSubLo);
    h[3] = h2_fma(((w >> 8) & 0x00F000F0u) | kMagic, kMulHi, kAddHi);
}
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t u4w(const uint4 &v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

constexpr int kMmaItemMax = 32;             // tokens of the largest mma.sync work item (4 n8 tiles)
constexpr int kMmaKB = 128;                 // reduction elements per ring stage (a multiple of 128)
constexpr int kMmaSub = kMmaKB / 128;       // 128-element sub-blocks per stage
constexpr int kMmaStages = 4;               // stages in the shared-memory ring
constexpr int kMmaARows = 256;              // weight rows per block (GU: 128 gate + 128 up)
constexpr int kMmaARowB = kMmaKB / 2;       // bytes of one weight row per stage (int4)
constexpr int kMmaABytes = kMmaARows * kMmaARowB;
constexpr int kMmaBLd = kMmaKB + 8;         // f16 per staged activation row (+ 8: no bank conflicts)
constexpr int kMmaBPieces = kMmaKB / 8;     // 16-byte copies per activation row per stage
constexpr int kMmaBBytes = kMmaItemMax * kMmaBLd * 2;
constexpr int kMmaStageBytes = kMmaABytes + kMmaBBytes;
constexpr size_t kMmaSmem = (size_t)kMmaStages * kMmaStageBytes;

__device__ __forceinline__ uint32_t smem_u32(const void *ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t lds32_u(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128_u(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// 8 signed int8 weights e0..e7 (bytes of lo = e0..e3, hi = e4..e7) -> the f16x2 pairs
// (e0,e4), (e1,e5), (e2,e6), (e3,e7), exact: the byte with its sign bit flipped is
// e + 128 in [0, 255], so 0x6400 | (e + 128) is the f16 1024 + e + 128; subtract 1152.
__device__ __forceinline__ void int8x8_to_f16x2(uint32_t lo, uint32_t hi, uint32_t (&h)[4]) {
    constexpr uint32_t kMagic = 0x64006400u;   // f16 1024 in both halves
    constexpr uint32_t kSub = 0x64806480u;     // 1152 = 1024 + 128
    lo ^= 0x80808080u;
    hi ^= 0x80808080u;
    h[0] = h2_sub((__byte_perm(lo, hi, 0x0400) & 0x00FF00FFu) | kMagic, kSub);
    h[1] = h2_sub((__byte_perm(lo, hi, 0x0501) & 0x00FF00FFu) | kMagic, kSub);
    h[2] = h2_sub((__byte_perm(lo, hi, 0x0602) & 0x00FF00FFu) | kMagic, kSub);
    h[3] = h2_sub((__byte_perm(lo, hi, 0x0703) & 0x00FF00FFu) | kMagic, kSub);
}

// Per-format layout of the weight half of a ring stage.  int4: a row's stage segment is
// kMmaKB / 2 bytes, stored unpadded (16-byte reads of rows 64 bytes apart are
// conflict-free); int8: kMmaKB bytes, rows padded by 16 bytes (a 128-byte stride would put
// a warp's eight rows on the same banks); two stages only, so both fit one allocation.
// Affine group-64 (G64): the int4 layout plus each row's float16 (scale, bias) pairs of the
// stage's groups (8 bytes per row per 128 elements) after the activations; three stages.
template <int FMT>
struct MmaFmt {
    static constexpr int kRowB = FMT == MOE_FORMAT_INT8 ? kMmaKB : kMmaKB / 2;   // global bytes per row
    static constexpr int kSRow = FMT == MOE_FORMAT_INT8 ? kRowB + 16 : kRowB;     // shared stride
    static constexpr int kPcs = kRowB / 16;                                      // 16-byte pieces per row
    static constexpr int kABytes = kMmaARows * kSRow;
    static constexpr int kSBRow = FMT == MOE_FORMAT_G64 ? kMmaKB / 64 * 4 : 0;  // group pairs per row
    static constexpr int kSBOff = kABytes + kMmaBBytes;
    static constexpr int kStage = kSBOff + kMmaARows * kSBRow;
    static constexpr int kStages = FMT == MOE_FORMAT_INT8 ? 2 : (FMT == MOE_FORMAT_G64 ? 3 : kMmaStages);
    static constexpr int kThrB = FMT == MOE_FORMAT_INT8 ? 32 : 16;               // a thread's bytes per row per sub-block
};
static_assert((size_t)MmaFmt<MOE_FORMAT_INT8>::kStages * MmaFmt<MOE_FORMAT_INT8>::kStage <= kMmaSmem,
              "the int8 ring fits the int4 ring's shared memory");
static_assert((size_t)MmaFmt<MOE_FORMAT_G64>::kStages * MmaFmt<MOE_FORMAT_G64>::kStage <= kMmaSmem,
              "the group-64 ring fits the int4 ring's shared memory");
static_assert(kMmaKB == 128, "the group-64 pairs of a stage are staged as one 8-byte copy per row");

__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

// 8 packed unsigned nibbles (element 2j in the low nibble) -> f16x2 pairs of u in [0, 15],
// (e0,e4), (e1,e5), (e2,e6), (e3,e7), exact; then w = s u + b, one f16 rounding.
__device__ __forceinline__ void g64x8_to_f16x2(uint32_t w, uint32_t s2, uint32_t b2, uint32_t (&h)[4]) {
    constexpr uint32_t kMagic = 0x64006400u;   // f16 1024
    constexpr uint32_t kMulHi = 0x2C002C00u;   // 1/16
    constexpr uint32_t kAddHi = 0xD400D400u;   // -64 = -1024/16
    h[0] = h2_fma(h2_sub((w & 0x000F000Fu) | kMagic, kMagic), s2, b2);
    h[1] = h2_fma(h2_fma((w & 0x00F000F0u) | kMagic, kMulHi, kAddHi), s2, b2);
    h[2] = h2_fma(h2_sub(((w >> 8) & 0x000F000Fu) | kMagic, kMagic), s2, b2);
    h[3] = h2_fma(h2_fma(((w >> 8) & 0x00F000F0u) | kMagic, kMulHi, kAddHi), s2, b2);
}

// One work item times one tile of output rows (see mma_expert_kernel), weights in format FMT.
template <bool GU, int FMT, int NT>
__device__ __forceinline__ void mma_body(const Params &p, int T, const SlotInfo &s, int nt, int o0,
                                         unsigned char *mma_smem, const int *s_brow, const int *s_orow) {
    using F = MmaFmt<FMT>;
    constexpr int kMmaNT = NT / 8;                     // n8 tiles of a work item
    const int H = p.d.H, Is = s.Is;
    const int rows = GU ? Is : H;                       // output rows of the slot
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
    const int Kd = GU ? H : Is;                          // reduction length
    const size_t arb = FMT == MOE_FORMAT_INT8 ? (size_t)Kd : (size_t)(Kd >> 1);   // weight row bytes
    const uint8_t *abase = GU ? s.slab : s.slab + 2 * (size_t)Is * (FMT == MOE_FORMAT_INT8 ? H : H >> 1);
    const uint16_t *act = GU ? p.ws.x16 : p.ws.h16;
    const size_t ald = GU ? (size_t)H : (size_t)p.d.I_max;     // activation row stride (f16)
    // this thread's cp.async pieces of one stage
    constexpr int kAP = F::kPcs, kBP = NT * kMmaBPieces / kThreads;   // copies per thread
    const uint8_t *asrc[kAP];
    uint32_t adst[kAP];
    int apiece[kAP];
    bool aok[kAP];
#pragma unroll
    for (int i = 0; i < kAP; i++) {
        const int c = tid + i * kThreads, lr = c / F::kPcs, piece = c % F::kPcs;
        const int gr = GU ? (lr < 128 ? o0 + lr : Is + o0 + lr - 128) : o0 + lr;
        aok[i] = GU || gr < H;
        apiece[i] = piece;
        asrc[i] = abase + (size_t)(aok[i] ? gr : 0) * arb + piece * 16;
        adst[i] = (uint32_t)(lr * F::kSRow + piece * 16);
    }
    const uint16_t *bsrc[kBP];
    uint32_t bdst[kBP];
    int bpiece[kBP];
    bool bok[kBP];                                 // rows of n8 tiles that are computed
#pragma unroll
    for (int i = 0; i < kBP; i++) {
        const int c = tid + i * kThreads, n = c / kMmaBPieces, piece = c % kMmaBPieces;
        bok[i] = n < ((nt + 7) & ~7);
        bpiece[i] = piece;
        bsrc[i] = act + (size_t)s_brow[n < nt ? n : 0] * ald + piece * 8;
        bdst[i] = (uint32_t)(F::kABytes + (n * kMmaBLd + piece * 8) * 2);
    }
    // G64: this thread copies the stage's (scale, bias) pairs of weight row `tid`
    const uint32_t *pbsrc = nullptr;
    bool pbok = false;
    if constexpr (FMT == MOE_FORMAT_G64) {
        const int lr = tid, gr = GU ? (lr < 128 ? o0 + lr : Is + o0 + lr - 128) : o0 + lr;
        pbok = GU || gr < H;
        const uint32_t *pairs = reinterpret_cast<const uint32_t *>(s.sc);
        pbsrc = GU ? pairs + (size_t)(pbok ? gr : 0) * (Kd / 64)
                   : pairs + 2 * (size_t)Is * (H / 64) + (size_t)(pbok ? gr : 0) * (Is / 64);
    }
    const uint32_t sbase = smem_u32(mma_smem);
    const int nkb = (Kd + kMmaKB - 1) / kMmaKB;     // the last stage may hold fewer sub-blocks
    auto issue = [&](int kb) {
        const uint32_t st = sbase + (uint32_t)((kb % F::kStages) * F::kStage);
        const int valid = min(kMmaKB, Kd - kb * kMmaKB);   // elements of this stage
        constexpr int kElemPerPiece = FMT == MOE_FORMAT_INT8 ? 16 : 32;
#pragma unroll
        for (int i = 0; i < kAP; i++)
            if (aok[i] && apiece[i] * kElemPerPiece < valid)
                cp_async16(st + adst[i], asrc[i] + (size_t)kb * F::kRowB);
#pragma unroll
        for (int i = 0; i < kBP; i++)
            if (bok[i] && bpiece[i] * 8 < valid) cp_async16(st + bdst[i], bsrc[i] + (size_t)kb * kMmaKB);
        if constexpr (FMT == MOE_FORMAT_G64) {
            if (pbok) cp_async8(st + F::kSBOff + tid * 8, pbsrc + (size_t)kb * (kMmaKB / 64));
        }
    };
    const int ob = o0 + (GU ? 16 : 32) * warp;            // the warp's first output row
    const bool active = ob < rows;                         // (rows are multiples of 128)
    // shared-memory offsets of the warp's four weight rows (tile 0 rows g, g+8; tile 1 rows g, g+8)
    uint32_t aoff[4];
    {
        const int l0 = GU ? 16 * warp + g : 32 * warp + g;
        const int l1 = GU ? 128 + 16 * warp + g : 32 * warp + 16 + g;
        aoff[0] = (uint32_t)(l0 * F::kSRow + q * F::kThrB);
        aoff[1] = aoff[0] + 8 * F::kSRow;
        aoff[2] = (uint32_t)(l1 * F::kSRow + q * F::kThrB);
        aoff[3] = aoff[2] + 8 * F::kSRow;
    }
    uint32_t sboff[4] = {0u, 0u, 0u, 0u};     // G64: the row's pair of the thread's group (q / 2)
    if constexpr (FMT == MOE_FORMAT_G64) {
        const int l0 = GU ? 16 * warp + g : 32 * warp + g;
        const int l1 = GU ? 128 + 16 * warp + g : 32 * warp + 16 + g;
        sboff[0] = (uint32_t)(F::kSBOff + l0 * 8 + (q >> 1) * 4);
        sboff[1] = sboff[0] + 8 * 8;
        sboff[2] = (uint32_t)(F::kSBOff + l1 * 8 + (q >> 1) * 4);
        sboff[3] = sboff[2] + 8 * 8;
    }
    uint32_t boff[kMmaNT];
#pragma unroll
    for (int j = 0; j < kMmaNT; j++) boff[j] = (uint32_t)(F::kABytes + ((8 * j + g) * kMmaBLd + 32 * q) * 2);
    const int ntiles = (nt + 7) >> 3;
    float acc[2][kMmaNT][4];
#pragma unroll
    for (int t = 0; t < 2; t++)
#pragma unroll
        for (int j = 0; j < kMmaNT; j++)
#pragma unroll
            for (int c = 0; c < 4; c++) acc[t][j][c] = 0.0f;
#pragma unroll
    for (int k = 0; k < F::kStages - 1; k++) {
        if (k < nkb) issue(k);
        cp_async_commit();
    }
#pragma unroll 1
    for (int kb = 0; kb < nkb; kb++) {
        cp_async_wait<F::kStages - 2>();     // this thread's pieces of stage kb have landed
        __syncthreads();                     // everyone's have; everyone is done with kb - 1
        if (kb + F::kStages - 1 < nkb) issue(kb + F::kStages - 1);
        cp_async_commit();
        if (!active) continue;
        const uint32_t st = sbase + (uint32_t)((kb % F::kStages) * F::kStage);
        const int nsub = min(kMmaSub, (Kd - kb * kMmaKB) >> 7);
#pragma unroll
        for (int sb = 0; sb < kMmaSub; sb++) {       // 128-element sub-blocks of the stage
            if (sb >= nsub) break;
            constexpr int kW = FMT == MOE_FORMAT_INT8 ? 2 : 1;     // 16-byte reads per row
            uint4 a[4][kW];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int r = 0; r < kW; r++) a[i][r] = lds128_u(st + aoff[i] + F::kThrB * 4 * sb + 16 * r);
            uint32_t s2[4] = {0u, 0u, 0u, 0u}, b2[4] = {0u, 0u, 0u, 0u};   // G64: (s, s) and (b, b)
            if constexpr (FMT == MOE_FORMAT_G64) {
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const uint32_t pr = lds32_u(st + sboff[i]);
                    s2[i] = __byte_perm(pr, pr, 0x1010);
                    b2[i] = __byte_perm(pr, pr, 0x3232);
                }
            }
#pragma unroll
            for (int w = 0; w < 4; w++) {        // group w: k-steps 2w (pairs 0, 1) and 2w + 1 (pairs 2, 3)
                uint32_t h[4][4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    if constexpr (FMT == MOE_FORMAT_INT8) {   // words 2w, 2w + 1 of the 32 bytes
                        const uint4 &v = a[i][w >> 1];
                        int8x8_to_f16x2(u4w(v, (2 * w) & 3), u4w(v, (2 * w + 1) & 3), h[i]);
                    } else if constexpr (FMT == MOE_FORMAT_G64) {
                        g64x8_to_f16x2(u4w(a[i][0], w), s2[i], b2[i], h[i]);
                    } else {
                        int4x8_to_f16x2(u4w(a[i][0], w), h[i]);
                    }
                }
#pragma unroll
                for (int j = 0; j < kMmaNT; j++)
                    if (j < ntiles) {
                        const uint4 b = lds128_u(st + boff[j] + 256 * sb + 16 * w);
#pragma unroll
                        for (int ss = 0; ss < 2; ss++) {
                            const int lo = 2 * ss, hi = 2 * ss + 1;
                            const uint32_t b0 = u4w(b, lo), b1 = u4w(b, hi);
                            mma_f16(acc[0][j], h[0][lo], h[1][lo], h[0][hi], h[1][hi], b0, b1);
                            mma_f16(acc[1][j], h[2][lo], h[3][lo], h[2][hi], h[3][hi], b0, b1);
                        }
                    }
            }
        }
    }
    cp_async_wait<0>();
    if (!active) return;
    // accumulator (tile t, n-tile j, c): row g + 8 (c >> 1) of the tile, token 8 j + 2 q + (c & 1)
    if (GU) {
#pragma unroll
        for (int rh = 0; rh < 2; rh++) {
            const int o = ob + g + 8 * rh;
            const float sg = FMT == MOE_FORMAT_G64 ? 1.0f : s.sc[o];     // G64: scales already applied
            const float su = FMT == MOE_FORMAT_G64 ? 1.0f : s.sc[Is + o];
            const int pos = mma_pos(o);
#pragma unroll
            for (int j = 0; j < kMmaNT; j++)
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    const int n = 8 * j + 2 * q + c;
                    if (j < ntiles && n < nt) {
                        const float hv = silu_mul(sg * acc[0][j][2 * rh + c], su * acc[1][j][2 * rh + c]);
                        p.ws.h16[(size_t)s_orow[n] * p.d.I_max + pos] = f2h_bits(hv);
                    }
                }
        }
    } else {
        const float *sd = s.sc + 2 * Is;
#pragma unroll
        for (int t = 0; t < 2; t++)
#pragma unroll
            for (int rh = 0; rh < 2; rh++) {
                const int o = ob + 16 * t + g + 8 * rh;
                const float sc = FMT == MOE_FORMAT_G64 ? 1.0f : sd[o];
#pragma unroll
                for (int j = 0; j < kMmaNT; j++)
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        const int n = 8 * j + 2 * q + c;
                        if (j < ntiles && n < nt) p.ws.dbuf[(size_t)s_orow[n] * H + o] = sc * acc[t][j][2 * rh + c];
                    }
            }
    }
}

// One work item times one tile of output rows.  GU (gate/up + SwiGLU): warp w
// owns output rows o0 + 16 w + {0..15}, as two m16 tiles: those gate rows and
// the same up rows; 128 rows per block; writes h16.  Down: warp w owns rows
// o0 + 32 w + {0..31} (two m16 tiles), 256 rows per block; writes dbuf.
// Weights (256 rows per stage) and the item's activations (NT rows)
// move through a ring in shared memory with cp.async; every stage is one
// __syncthreads.  FR / FS: weight formats of the routed experts / the shared
// expert; each instantiation carries only the bodies it needs, so a config with
// one format gets the lean kernel and a mixed one still runs in one launch.
template <bool GU, int FR, int FS, int NT>
__global__ void __launch_bounds__(kThreads, 2) mma_expert_kernel(Params p, int T) {
    extern __shared__ __align__(128) unsigned char mma_smem[];
    __shared__ int s_brow[NT], s_orow[NT];
    const int item = blockIdx.x;
    if (item >= *p.ws.n_items) return;
    const int slot = p.ws.items[2 * item], n0 = p.ws.items[2 * item + 1];
    const SlotInfo s = slot_info(p, T, slot);
    if (!s.valid) return;
    const int o0 = blockIdx.y * (GU ? 128 : 256);
    if (o0 >= (GU ? s.Is : p.d.H)) return;
    const int tid = threadIdx.x;
    const int nt = min(NT, s.n - n0);
    if (tid < NT) {
        int tok = 0, row = -1;
        if (tid < nt) slot_token(p, s, T, n0 + tid, &tok, &row);
        s_brow[tid] = GU ? tok : row;          // activation row the tensor cores read
        s_orow[tid] = row;                     // output row (h16 / dbuf)
    }
    __syncthreads();
    if (FR == FS || s.base >= 0)
        mma_body<GU, FR, NT>(p, T, s, nt, o0, mma_smem, s_brow, s_orow);
    else
        mma_body<GU, FS, NT>(p, T, s, nt, o0, mma_smem, s_brow, s_orow);
}

// ---------------------------------------------------------------------------
// Batched (T > 1) int4 experts on the 5th-generation tensor cores (tcgen05.mma,
// accumulators in tensor memory).
//
// One block = one work item (a slot and up to kTcTok of its tokens) x kTcTiles
// 128-row weight tiles (gate/up: the gate rows and the up rows of 128 outputs;
// down: 256 output rows), one 128 x 128 f32 accumulator each in tensor memory.
// Measured on this GPU, one M 128 x K 16 MMA occupies the SM's tensor core
// ~33-36 ns for any N up to 128, so the items are 128 tokens wide.  The
// reduction runs in stages of kTcKB elements, each warp with one role:
//   warps 0, 1   issue the MMAs of tile 0 / 1 (one thread each, in stage order,
//                so every accumulator sums in a fixed order) with A, the
//                dequantised weights, in tensor memory and B, the activations,
//                in shared memory; each stage's two commits free its slots;
//   warp 2       copies the block's raw int4 rows, two stages at a time, by 2-D
//                tensor copies (64-byte rows, 64-byte swizzle) into a kTcR-slot
//                ring;
//   warp 3       copies a stage's activations, already in the operand layout
//                (tc_act_index), by one contiguous bulk copy into a kTcS-slot ring;
//   warps 4-11   dequantise: thread = weight row, 64 int4 of a stage -> 32 f16
//                pairs -> tcgen05.st into the stage's A columns (lane = row, column
//                c = the pair of K positions 2c, 2c + 1).
// Full/empty mbarriers connect the roles.  The issuing thread's code between MMAs
// is kept to one 64-bit add (measured: a single thread issues at the tensor
// core's rate only when descriptors are precomputed).  Operands are K-major
// without swizzle: core matrices of 8 rows x 16 bytes; the K order inside every
// 8-element group is the mma order of the activations (0 4 1 5 2 6 3 7), exactly
// the order of int4x8_to_f16x2's pairs.  Every wait is bounded; a block that
// gives up sets kErrTc, waits (bounded) for its copies in flight and its MMAs,
// and still frees its tensor memory.
// ---------------------------------------------------------------------------

constexpr int kTcTok = 128;                        // tokens of a work item on this path (MMA N)
constexpr int kTcTiles = 2;                        // 128-row weight tiles per block (one accumulator each)
constexpr int kTcRows = 128 * kTcTiles;            // weight rows per block (gate/up: the gate and up rows of 128 outputs)
constexpr int kTcKB = 64;                          // reduction elements per stage
constexpr int kTcS = 4;                            // stage slots: activations (shared memory) and A (tensor memory)
constexpr int kTcRawB = 64;                        // bytes of a weight row per tensor copy (two stages)
constexpr int kTcR = 8;                            // raw ring slots (two stages each)
constexpr int kTcBGroup = kTcTok * 16;             // activations: one 8-element k-group of the item's rows
constexpr int kTcBTile = kTcBGroup * (kTcKB / 8);  // the item's f16 activations of a stage (one copy)
constexpr int kTcRawBox = 128;                     // weight rows of one tensor copy (box height)
constexpr int kTcRawSlot = kTcRows * kTcRawB;      // the block's int4 rows of two stages
constexpr int kTcACols = kTcTiles * (kTcKB / 2);   // A columns per stage (two f16 per 32-bit column)
constexpr int kTcCols = 512;                       // allocation: accumulators + the A ring
constexpr int kTcDq0 = 4;                          // warps: 0, 1 MMA (tile 0, 1), 2 weight copies, 3 activation copies, 4.. dequant
constexpr int kTcWarps = kTcDq0 + kTcRows / 32;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr size_t kTcSmem = (size_t)kTcS * kTcBTile + (size_t)kTcR * kTcRawSlot + 1024;
constexpr unsigned kErrTc = MOE_DEVICE_ERR_TC;
// kind::f16: D f32 (bits 4-5 = 1), A and B f16 (0), both K-major (0), N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t kTcIdesc = (1u << 4) | ((uint32_t)(kTcTok >> 3) << 17) | ((128u >> 4) << 24);
constexpr unsigned long long kTcWaitNs = 500ull * 1000 * 1000;
static_assert(kTcSmem + 1024 <= 227 * 1024, "both rings and the static arrays fit one block's shared memory");
static_assert(kTcTiles == 2, "one MMA-issuing warp per tile: warps 0 and 1");
static_assert(kTcTiles * kTcTok + kTcS * kTcACols <= kTcCols, "accumulators and the A ring fit the allocation");
static_assert(kTcRawB == 2 * (kTcKB / 2) && kTcRawSlot == 2 * kTcRawBox * kTcRawB, "a raw slot is two copies of two stages");
static_assert(kTcRows / 32 == 8 && kTcDq0 % 4 == 0, "eight dequantising warps cover each lane quarter of each tile once");

// no-swizzle K-major operand descriptor: core matrices of 8 rows x 16 bytes, lbo bytes apart
// along K, sbo bytes apart per 8 rows
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long tc_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// wait (bounded) for phase `parity` of an mbarrier; false when the wait ran out
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = tc_now();
    for (;;) {
        for (int i = 0; i < 64; i++)
            if (mbar_try(bar, parity)) return true;
        if (tc_now() - t0 > kTcWaitNs) return false;
    }
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// this thread's arrival, announcing `bytes` of tensor copies that complete the phase
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// 2-D tensor copy global -> shared (box of the tensor map at element x, row y; rows outside the
// tensor read as zeros), counted on the mbarrier
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, int x, int y, uint32_t bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar) : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void tc_mma_ta(uint32_t dtaddr, uint32_t ataddr, uint64_t bd, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(dtaddr), "r"(ataddr), "l"(bd), "r"(kTcIdesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                   "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
                   "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
                   "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
// contiguous copy global -> shared (16-byte aligned, a multiple of 16 bytes), counted on the mbarrier
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// The tcgen05 path's activations, [stage][item][k-group][row][8 f16]: one stage (kTcKB elements)
// of one work item's kTcTok rows is one contiguous kTcBTile block, already in the operand layout
// (k-group j at j kTcBGroup, row n at 16 n).  Gate/up reads xp16 (written by permute_x16_kernel);
// down reads h16 (written by the gate/up epilogue of the same item).
__device__ __forceinline__ size_t tc_act_index(int stage, int item, int cap) {   // in f16 elements
    return ((size_t)stage * (size_t)cap + (size_t)item) * (size_t)(kTcBTile / 2);
}

template <bool GU>
__global__ void __launch_bounds__(kTcThreads, 1) tc_expert_kernel(Params p, int T) {
    extern __shared__ __align__(1024) unsigned char tc_smem[];
    __shared__ int s_orow[kTcTok];
    __shared__ __align__(8) unsigned long long s_rfull[kTcR];   // a raw slot's int4 rows have landed
    __shared__ __align__(8) unsigned long long s_rempty[kTcR];  // the dequantising warps are done with a raw slot
    __shared__ __align__(8) unsigned long long s_bfull[kTcS];   // a stage's activation copy has landed
    __shared__ __align__(8) unsigned long long s_full[kTcS];    // a stage's A columns are written (eight warps)
    __shared__ __align__(8) unsigned long long s_mdone[kTcS];   // a stage's MMAs of both tiles are done (two commits)
    __shared__ __align__(8) unsigned long long s_drain[kTcTiles];   // all MMAs an issuing thread made are done
    __shared__ uint32_t s_taddr;
    __shared__ int s_fail;
    __shared__ int s_r_issued, s_b_issued;   // for the bounded drain after a failure
    const int item = blockIdx.y;      // row blocks of one item run together: its activations and
                                       // (items of one expert are adjacent) its weights stay in L2
    if (item >= *p.ws.n_items) return;
    const int slot = p.ws.items[2 * item], n0 = p.ws.items[2 * item + 1];
    const SlotInfo s = slot_info(p, T, slot);
    if (!s.valid) return;
    const int H = p.d.H, Is = s.Is;
    const int rows = GU ? Is : H;
    const int o0 = blockIdx.x * (GU ? kTcRows / 2 : kTcRows);
    if (o0 >= rows) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = min(kTcTok, s.n - n0);
    if (tid < kTcTok) {
        int tok = 0, row = -1;
        if (tid < nt) slot_token(p, s, T, n0 + tid, &tok, &row);
        s_orow[tid] = row;
    }
    if (tid == 0) {
        s_fail = 0;
        s_r_issued = -1;
        s_b_issued = -1;
        for (int i = 0; i < kTcR; i++) {
            mbar_init(smem_u32(&s_rfull[i]), 1);
            mbar_init(smem_u32(&s_rempty[i]), kTcRows / 32);
        }
        for (int i = 0; i < kTcS; i++) {
            mbar_init(smem_u32(&s_bfull[i]), 1);
            mbar_init(smem_u32(&s_full[i]), kTcRows / 32);
            mbar_init(smem_u32(&s_mdone[i]), kTcTiles);
        }
        for (int i = 0; i < kTcTiles; i++) mbar_init(smem_u32(&s_drain[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&s_taddr)), "n"(kTcCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = s_taddr;
    volatile int *fail = &s_fail;

    const int Kd = GU ? H : Is;
    const int nkb = Kd / kTcKB, nq = Kd / (2 * kTcRawB);
    const int cap = p.ws.tc_items;
    const uint32_t sbase = (smem_u32(tc_smem) + 1023u) & ~1023u;
    const uint32_t rbase = sbase + (uint32_t)(kTcS * kTcBTile);
    if (warp < kTcTiles) {
        // MMA issue, tile t = warp: stage kb once its A columns and activations are in; the two
        // tiles' commits together free the stage's slots.  Each tile accumulates in stage order.
        if (lane == 0) {
            const int t = warp;
            bool issued = false;
            // everything but the slot is fixed: the B descriptor of slot j and k-step ks is the
            // slot-0 descriptor plus the byte offset / 16 in its start-address field (shared
            // addresses stay below 2^18, so the field cannot carry), the A column likewise
            const uint64_t bd0 = tc_desc(sbase, kTcBGroup, 128);
            const uint32_t dt = taddr + (uint32_t)(kTcTok * t);
            const uint32_t at0 = taddr + (uint32_t)(kTcTiles * kTcTok + t * (kTcKB / 2));
            for (int kb = 0; kb < nkb; kb++) {
                if (*fail) break;
                const int j = kb % kTcS;
                const uint64_t bd = bd0 + (uint64_t)((j * kTcBTile) >> 4);
                const uint32_t at = at0 + (uint32_t)(j * kTcACols);
                if (!mbar_wait(smem_u32(&s_full[j]), (uint32_t)(kb / kTcS) & 1u) ||
                    !mbar_wait(smem_u32(&s_bfull[j]), (uint32_t)(kb / kTcS) & 1u)) {
                    *fail = 1;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                tc_mma_ta(dt, at, bd, kb > 0 ? 1u : 0u);      // K 16 per MMA: 8 A columns, two k-groups of B
#pragma unroll
                for (int ks = 1; ks < kTcKB / 16; ks++)
                    tc_mma_ta(dt, at + (uint32_t)(8 * ks), bd + (uint64_t)((2 * kTcBGroup * ks) >> 4), 1u);
                tc_commit(smem_u32(&s_mdone[j]));
                issued = true;
            }
            // every MMA this thread issued is done before the block moves on (bounded)
            if (issued) {
                tc_commit(smem_u32(&s_drain[t]));
                if (!mbar_wait(smem_u32(&s_drain[t]), 0u)) *fail = 1;
            }
        }
    } else if (warp == kTcTiles) {
        // weight copies: raw slot q % kTcR (stages 2q, 2q + 1 of the block's rows) once the
        // dequantising warps are done with its previous use
        if (lane == 0) {
            const int me = s.base >= 0 ? p.ws.slot_expert[slot] : p.d.E;
            const void *wmap = static_cast<const unsigned char *>(p.tmaps) + (size_t)(2 * me + (GU ? 0 : 1)) * kTmapBytes;
            const int wy0 = o0, wy1 = GU ? Is + o0 : o0 + kTcRawBox;
            for (int q = 0; q < nq; q++) {
                if (*fail) break;
                if (q >= kTcR && !mbar_wait(smem_u32(&s_rempty[q % kTcR]), (uint32_t)((q - kTcR) / kTcR) & 1u)) {
                    *fail = 1;
                    break;
                }
                const uint32_t bar = smem_u32(&s_rfull[q % kTcR]);
                const uint32_t dst = rbase + (uint32_t)((q % kTcR) * kTcRawSlot);
                mbar_expect_tx(bar, kTcRawSlot);
                tma_load_2d(dst, wmap, q * kTcRawB, wy0, bar);
                tma_load_2d(dst + kTcRawBox * kTcRawB, wmap, q * kTcRawB, wy1, bar);
                s_r_issued = q;
            }
        }
    } else if (warp == kTcTiles + 1) {
        // activation copies: slot kb % kTcS once the MMAs of its previous use are done
        if (lane == 0) {
            const uint16_t *act = GU ? p.ws.xp16 : p.ws.h16;
            for (int kb = 0; kb < nkb; kb++) {
                if (*fail) break;
                if (kb >= kTcS && !mbar_wait(smem_u32(&s_mdone[kb % kTcS]), (uint32_t)((kb - kTcS) / kTcS) & 1u)) {
                    *fail = 1;
                    break;
                }
                const uint32_t bar = smem_u32(&s_bfull[kb % kTcS]);
                mbar_expect_tx(bar, kTcBTile);
                bulk_load(sbase + (uint32_t)((kb % kTcS) * kTcBTile), act + tc_act_index(kb, item, cap), kTcBTile, bar);
                s_b_issued = kb;
            }
        }
    } else {
        // dequantisation: thread = weight row r = 32 (warp % 4) + lane of tile t (the warp's own
        // tensor-memory lanes; gate/up: tile 0 the gate rows, tile 1 the up rows).  Raw rows are 64
        // bytes apart with the copy's 64-byte swizzle: 16-byte chunk c of row lr at c ^ ((lr >> 1) & 3).
        const int t = (warp - kTcDq0) >> 2;
        const int lr = t * 128 + 32 * (warp & 3) + lane;
        const uint32_t rrow = (uint32_t)(lr * kTcRawB), rsw = (uint32_t)((lr >> 1) & 3);
        const uint32_t tcol = taddr + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(kTcTiles * kTcTok + t * (kTcKB / 2));
        // this row's 64 values of stage k -> 32 f16 pairs (mma order), once its raw slot has landed;
        // false: the wait ran out (warp-uniform)
        uint32_t h32[32];
        auto convert = [&](int k) -> bool {
            const int q = k >> 1;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s_rfull[q % kTcR]), (uint32_t)(q / kTcR) & 1u)))
                return false;
            const uint32_t rs = rbase + (uint32_t)((q % kTcR) * kTcRawSlot) + rrow;
            const uint32_t c0 = (uint32_t)(2 * (k & 1));
            const uint4 wa = lds128(rs + ((c0 ^ rsw) << 4));
            const uint4 wb = lds128(rs + (((c0 + 1) ^ rsw) << 4));
            const uint32_t w8[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int m = 0; m < 8; m++) {
                uint32_t h[4];
                int4x8_to_f16x2(w8[m], h);
#pragma unroll
                for (int c = 0; c < 4; c++) h32[4 * m + c] = h[c];
            }
            if (k & 1) {                        // both stages of raw slot q are read
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s_rempty[q % kTcR]));
            }
            return true;
        };
        // stage kb: its pairs are already in registers; once the A slot's previous stage has been
        // consumed they go to tensor memory and the stage is reported, then stage kb + 1 is converted
        // (off the path from a commit to the next MMAs)
        bool ok = convert(0);
        if (!ok) *fail = 1;
        for (int kb = 0; kb < nkb && ok; kb++) {
            if (__any_sync(0xffffffffu, *fail != 0)) break;
            if (kb >= kTcS &&
                !__all_sync(0xffffffffu, mbar_wait(smem_u32(&s_mdone[kb % kTcS]), (uint32_t)((kb - kTcS) / kTcS) & 1u))) {
                *fail = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            tc_st32(tcol + (uint32_t)((kb % kTcS) * kTcACols), h32);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s_full[kb % kTcS]));
            if (kb + 1 < nkb && !convert(kb + 1)) {
                *fail = 1;
                break;
            }
        }
    }
    __syncthreads();
    if (s_fail && tid == 0) {
        // after a wait that ran out: copies still in flight land before the block's shared memory
        // is released (every wait bounded); the MMA threads already waited for their own MMAs
        for (int q = max(0, s_r_issued - kTcR + 1); q <= s_r_issued; q++)
            mbar_wait(smem_u32(&s_rfull[q % kTcR]), (uint32_t)(q / kTcR) & 1u);
        for (int k = max(0, s_b_issued - kTcS + 1); k <= s_b_issued; k++)
            mbar_wait(smem_u32(&s_bfull[k % kTcS]), (uint32_t)(k / kTcS) & 1u);
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (s_fail) {
        if (tid == 0) atomicOr(p.ws.err, kErrTc);
    } else if (warp >= kTcDq0) {
        // warp w: lane quarter w % 4; gate/up: tokens 64 hw .. + 63 of the gate tile and the up tile;
        // down: tile hw, all tokens (hw = 0 for warps 4-7, 1 for 8-11)
        const int q4 = warp & 3, hw = (warp - kTcDq0) >> 2;
        const uint32_t trow = taddr + ((uint32_t)(32 * q4) << 16);
        if (GU) {
            const int o = o0 + 32 * q4 + lane;     // gate row o and up row o
            const bool ok = o < Is;
            const float sg = ok ? s.sc[o] : 0.0f, su = ok ? s.sc[Is + o] : 0.0f;
            const int pos = mma_pos(o);
            // h of this item in the down kernel's activation layout: stage pos / kTcKB, k-group, element
            uint16_t *hp = p.ws.h16 + tc_act_index(pos / kTcKB, item, cap) + (size_t)((pos >> 3) & 7) * (kTcBGroup / 2) + (pos & 7);
#pragma unroll 1
            for (int c = 4 * hw; c < 4 * hw + kTcTok / 32; c++) {
                float g[16], u[16];
                tc_ld16(trow + 16 * c, g);
                tc_ld16(trow + kTcTok + 16 * c, u);
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const int n = 16 * c + i;
                    if (ok && n < nt) hp[n * 8] = f2h_bits(silu_mul(sg * g[i], su * u[i]));
                }
            }
        } else {
            const int o = o0 + 128 * hw + 32 * q4 + lane;
            const float sd = o < H ? s.sc[2 * Is + o] : 0.0f;
#pragma unroll 1
            for (int c = 0; c < kTcTok / 16; c++) {
                float v[16];
                tc_ld16(trow + kTcTok * hw + 16 * c, v);
                if (o < H) {
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int n = 16 * c + i;
                        if (n < nt) p.ws.dbuf[(size_t)s_orow[n] * H + o] = sd * v[i];
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kTcCols) : "memory");
}

// tcgen05 gate/up activations: xp16 holds, for every work item, the x16 rows of its tokens in the
// layout above (stage, item, k-group, row).  Block: one item x 32 of its rows x the k-groups of
// slice blockIdx.z; rows past the item's tokens stay unwritten (their accumulator columns are
// never read).
constexpr int kPermSlices = 8;
__global__ void __launch_bounds__(kThreads) permute_x16_kernel(Params p, int T) {
    const int item = blockIdx.x;
    if (item >= *p.ws.n_items) return;
    const int slot = p.ws.items[2 * item], n0 = p.ws.items[2 * item + 1];
    const SlotInfo s = slot_info(p, T, slot);
    if (!s.valid) return;
    const int n = blockIdx.y * 32 + (threadIdx.x & 31);
    if (n0 + n >= s.n) return;
    int tok = 0, row = 0;
    slot_token(p, s, T, n0 + n, &tok, &row);
    const int H = p.d.H, warp = threadIdx.x >> 5, cap = p.ws.tc_items;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.ws.x16 + (size_t)tok * H);
    uint4 *dst = reinterpret_cast<uint4 *>(p.ws.xp16);
    for (int g = blockIdx.z * kWarps + warp; g < H / 8; g += kWarps * kPermSlices)
        dst[(tc_act_index(g / (kTcKB / 8), item, cap) + (size_t)(g % (kTcKB / 8)) * (kTcBGroup / 2)) / 8 + n] =
            __ldcg(src + g);
}

template <bool GU, int FR, int FS>
cudaError_t mma_attr() {
    cudaError_t e = cudaFuncSetAttribute(mma_expert_kernel<GU, FR, FS, 16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMmaSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mma_expert_kernel<GU, FR, FS, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kMmaSmem);
    return e;
}

// The (routed, shared) format pair of a config as one switch value.
inline int fmt_pair(const Dims &d) { return d.expert_fmt * 3 + (d.n_shared ? d.shared_fmt : d.expert_fmt); }

#define MOE_FMT_PAIRS(X) X(0, 0) X(0, 1) X(0, 2) X(1, 0) X(1, 1) X(1, 2) X(2, 0) X(2, 1) X(2, 2)

constexpr bool kUseTc = true;   // int4 experts on tcgen05 for large T (else always the mma.sync kernel)
// tcgen05 from this many tokens per call: it wins where the 128-token items are full (measured
// on the GLM layer at T 512: gate/up 0.42 vs 0.78 ms, down 0.24 vs 0.40 ms against the mma.sync
// kernel; at T <= 64 the mma.sync kernel is faster)
constexpr int kTcMinT = 256;

// Tokens of a tensor-core work item for a call of T tokens: 128 on tcgen05; on the
// mma.sync kernel 16 while experts see few tokens each (measured on the GLM layer at
// T 16 and 64: gate/up and down ~22 % faster than with 32-token items), 32 once the mean
// routed expert gets 24 or more (OLMoE-shaped int8 layer at T 256: 32-token items 22 %
// faster, each expert's weights read half as often).
int mma_item_tokens(const Dims &d, int T) {
    if (d.tc && T >= kTcMinT) return kTcTok;
    return (long)T * d.K >= 24L * d.E ? kMmaItemMax : kItemTokens;
}

// Launch the tensor-core kernel of one phase (gate/up or down) for the config's formats.
template <bool GU>
void launch_mma_phase(const Params &p, int T, dim3 grid, cudaStream_t st) {
    if (p.item_tok == kTcTok) {
        const dim3 g(GU ? (p.d.I_max + kTcRows / 2 - 1) / (kTcRows / 2) : (p.d.H + kTcRows - 1) / kTcRows, grid.x);
        if (GU) permute_x16_kernel<<<dim3(grid.x, kTcTok / 32, kPermSlices), kThreads, 0, st>>>(p, T);
        tc_expert_kernel<GU><<<g, kTcThreads, kTcSmem, st>>>(p, T);
        return;
    }
    switch (fmt_pair(p.d)) {
#define MOE_LAUNCH(R, S)                                                                  \
    case R * 3 + S:                                                                       \
        if (p.item_tok == 32) mma_expert_kernel<GU, R, S, 32><<<grid, kThreads, kMmaSmem, st>>>(p, T); \
        else mma_expert_kernel<GU, R, S, 16><<<grid, kThreads, kMmaSmem, st>>>(p, T);    \
        break;
        MOE_FMT_PAIRS(MOE_LAUNCH)
#undef MOE_LAUNCH
    }
}

size_t router_smem_bytes(const Dims &d) {
    const size_t topk = (size_t)kWarps * 2 * d.E * sizeof(float);
    const size_t bucket = (size_t)(2 + kWarps) * d.E * sizeof(int);
    return topk > bucket ? topk : bucket;
}

// k-ranges of the tiled router for T tokens: about kRouterBlocks blocks in all
int router_split(int T, int E, int H) {
    const int tiles = ((E + kRtExp - 1) / kRtExp) * ((T + kRtTok - 1) / kRtTok);
    int S = kRouterBlocks / tiles;
    if (S > kRouterMaxSplit) S = kRouterMaxSplit;
    if (S > H / kRtK) S = H / kRtK;
    return S < 1 ? 1 : S;
}

// largest S * T of any tiled-router call up to maxT tokens (partial-logit rows)
size_t router_part_rows(const Dims &d) {
    size_t m = 0;
    for (int T = kGemvMaxT + 1; T <= d.max_tokens; T++) {
        const size_t v = (size_t)router_split(T, d.E, d.H) * (size_t)T;
        if (v > m) m = v;
    }
    return m;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

// ---------------------------------------------------------------------------
// Workspace
// ---------------------------------------------------------------------------

size_t workspace_bytes(const Dims &d) {
    Workspace ws;
    carve_workspace(d, nullptr, &ws);
    return ws.total_bytes;
}

void carve_workspace(const Dims &d, void *base, Workspace *ws) {
    char *b = static_cast<char *>(base);
    size_t o = 0;
    auto take = [&](size_t bytes) { char *r = b + o; o += align_up(bytes, 256); return r; };
    const size_t T = d.max_tokens, P = T * d.K;
    ws->rnorm = reinterpret_cast<float *>(take(T * sizeof(float)));
    ws->xperm = reinterpret_cast<float *>(take(T * d.H * sizeof(float)));
    ws->logits = reinterpret_cast<float *>(take(T * d.E * sizeof(float)));
    ws->topk_idx = reinterpret_cast<int *>(take(P * sizeof(int)));
    ws->topk_w = reinterpret_cast<float *>(take(P * sizeof(float)));
    ws->counters = reinterpret_cast<unsigned *>(take(16 * sizeof(unsigned)));
    ws->h = reinterpret_cast<float *>(take((P + T) * d.I_max * sizeof(float)));
    ws->cnt = reinterpret_cast<int *>(take(d.E * sizeof(int)));
    ws->off = reinterpret_cast<int *>(take((d.E + 1) * sizeof(int)));
    ws->perm = reinterpret_cast<int *>(take(P * sizeof(int)));
    ws->inv = reinterpret_cast<int *>(take(P * sizeof(int)));
    ws->slot_expert = reinterpret_cast<int *>(take(d.E * sizeof(int)));
    ws->n_slots = reinterpret_cast<int *>(take(sizeof(int)));
    ws->err = reinterpret_cast<unsigned *>(take(4 * sizeof(unsigned)));
    ws->dpart = reinterpret_cast<float *>(take((size_t)kMaxSlots * d.H * sizeof(float)));
    ws->dscore = reinterpret_cast<float *>(take(2 * (size_t)d.E * sizeof(float)));
    ws->trace = reinterpret_cast<unsigned long long *>(
        take(d.trace ? (size_t)kTraceBlocks * MOE_TRACE_SLOTS * sizeof(unsigned long long) : 0));
    ws->dbuf = reinterpret_cast<float *>(take((P + T) * d.H * sizeof(float)));
    const bool mma = d.mma != 0 && (T > 1 || d.mma_fmt);
    ws->x16 = reinterpret_cast<uint16_t *>(take(mma ? T * d.H * sizeof(uint16_t) : 0));
    // tcgen05 path: h16 and xp16 also in the item-blocked activation layout of tc_act_index
    // (tc_items work items of kTcTok rows); h16 is row-major on the other paths
    const bool tcp = tc_maps_needed(d);
    ws->tc_items = tcp ? max_items((int)T, d.K, d.E, d.n_shared, kTcTok) : 0;
    const size_t tc_h = (size_t)ws->tc_items * kTcTok * d.I_max, rm_h = (P + T) * d.I_max;
    ws->h16 = reinterpret_cast<uint16_t *>(take(!mma ? 0 : (tc_h > rm_h ? tc_h : rm_h) * sizeof(uint16_t)));
    ws->xp16 = reinterpret_cast<uint16_t *>(take((size_t)ws->tc_items * kTcTok * d.H * sizeof(uint16_t)));
    ws->items = reinterpret_cast<int *>(
        take(mma ? 2 * (size_t)max_items((int)T, d.K, d.E, d.n_shared) * sizeof(int) : 0));
    ws->n_items = reinterpret_cast<int *>(take(sizeof(int)));
    const bool tiled = T > (size_t)kGemvMaxT;
    const size_t prows = tiled ? router_part_rows(d) : 0;
    ws->lpart = reinterpret_cast<float *>(take(prows * d.E * sizeof(float)));
    ws->sspart = reinterpret_cast<float *>(take(prows * sizeof(float)));
    ws->total_bytes = o;
}

// ---------------------------------------------------------------------------
// Launch
// ---------------------------------------------------------------------------

bool tc_supported(const Dims &d) {
    const bool int4_only = d.expert_fmt == MOE_FORMAT_INT4 && (!d.n_shared || d.shared_fmt == MOE_FORMAT_INT4);
    return kUseTc && int4_only;
}

bool tc_maps_needed(const Dims &d) { return d.mma && d.tc && d.max_tokens >= kTcMinT; }

size_t tc_map_count(const Dims &d) { return tc_maps_needed(d) ? 2 * (size_t)d.E + 2 : 0; }

cudaError_t upload_tc_maps(const Params &p, const uint8_t *const *host_slabs, void *dev) {
    static_assert(sizeof(CUtensorMap) == kTmapBytes, "tensor-map size");
    const Dims &d = p.d;
    const size_t n = tc_map_count(d);
    if (n == 0) return cudaSuccess;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    std::vector<CUtensorMap> m(n);
    std::memset(m.data(), 0, n * sizeof(CUtensorMap));
    // weights, uint8 [rows, cols]: boxes of kTcRawB bytes (two stages) x kTcRawBox rows, stored with
    // the 64-byte swizzle (16-byte chunk c of box row r at chunk c ^ ((r >> 1) & 3)); rows past the
    // tensor read as zeros.  Gate/up: rows [0, 2 Is) of H / 2 bytes; down: rows [0, H) of Is / 2
    // bytes after them.
    bool ok = true;
    auto map2d = [&](size_t i, const void *base, uint64_t cols, uint64_t rows) {
        const cuuint64_t dims[2] = {cols, rows};
        const cuuint64_t strides[1] = {cols};
        const cuuint32_t box[2] = {(cuuint32_t)kTcRawB, (cuuint32_t)kTcRawBox};
        const cuuint32_t es[2] = {1, 1};
        ok = ok && encode(&m[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    auto weights = [&](size_t i, const uint8_t *slab, int Is) {
        map2d(2 * i, slab, (uint64_t)d.H / 2, 2 * (uint64_t)Is);
        map2d(2 * i + 1, slab + (size_t)Is * d.H, (uint64_t)Is / 2, (uint64_t)d.H);
    };
    for (int x = 0; x < d.E; x++)
        if (host_slabs[x]) weights((size_t)x, host_slabs[x], d.I);
    if (d.n_shared) weights((size_t)d.E, p.sh_slab, d.I_sh);
    if (!ok) return cudaErrorInvalidValue;
    return cudaMemcpy(dev, m.data(), n * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
}

bool mma_supported(const Dims &d) {
    return (d.max_tokens > 1 || d.mma_fmt) && d.H % 128 == 0 && d.I % 128 == 0 &&
           (!d.n_shared || d.I_sh % 128 == 0);
}

cudaError_t prepare_kernels(Dims &d) {
    const int smem = (int)router_smem_bytes(d);
    cudaError_t e = cudaFuncSetAttribute(router_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(router_tiled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRtSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(router_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess && d.mma && d.tc) {
        e = cudaFuncSetAttribute(tc_expert_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc_expert_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    }
    if (e == cudaSuccess && d.mma) {
        switch (fmt_pair(d)) {
#define MOE_ATTR(R, S) \
    case R * 3 + S: e = mma_attr<true, R, S>(); if (e == cudaSuccess) e = mma_attr<false, R, S>(); break;
            MOE_FMT_PAIRS(MOE_ATTR)
#undef MOE_ATTR
        }
    }
    if (e == cudaSuccess && d.fast_decode) e = prepare_decode_fast(d);
    return e;
}

// ---------------------------------------------------------------------------
// Checked build (MOE_FLAG_DEBUG_CHECKS): routing and bucket invariants of a call
// ---------------------------------------------------------------------------

constexpr unsigned kErrCheck = MOE_DEVICE_ERR_CHECK;

// One block.  Every index is range-checked before it is used as an address, so
// any workspace contents are safe to check.  A failure ORs kErrCheck into
// err[0] and records (pair + 1, code) in err[1], err[2] (the first to claim).
__global__ void __launch_bounds__(kThreads) check_kernel(Params p, int T, int buckets) {
    const int K = p.d.K, E = p.d.E, P = T * K;
    const int *idx = p.ws.topk_idx;
    __shared__ int s_owned;
    if (threadIdx.x == 0) s_owned = 0;
    __syncthreads();
    auto fail = [&](int where, int code) {
        atomicOr(p.ws.err, kErrCheck);
        if (atomicCAS(p.ws.err + 1, 0u, (unsigned)where + 1u) == 0u) p.ws.err[2] = (unsigned)code;
    };
    int owned = 0;
    for (int q = threadIdx.x; q < P; q += blockDim.x) {
        const int e = idx[q];
        if (e < 0 || e >= E) { fail(q, 1); continue; }
        if (!isfinite(p.ws.topk_w[q])) fail(q, 2);
        const int t0 = q - q % K;
        for (int q2 = t0; q2 < q; q2++)
            if (idx[q2] == e) fail(q, 3);
        if (!buckets) continue;
        const bool own = e >= p.d.ep_lo && e < p.d.ep_hi;
        const int pos = p.ws.inv[q];
        if (!own) {
            if (pos != -1) fail(q, 4);
            continue;
        }
        owned++;
        const int lo = p.ws.off[e], hi = p.ws.off[e + 1];
        if (pos < 0 || pos >= P || pos < lo || pos >= hi || p.ws.perm[pos] != q) fail(q, 5);
    }
    if (!buckets) return;
    atomicAdd(&s_owned, owned);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = p.ws.cnt[e], lo = p.ws.off[e], hi = p.ws.off[e + 1];
        if (c < 0 || hi - lo != c || (e == 0 && lo != 0) || hi > P) fail(P + e, 6);
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.ws.off[E] != s_owned) fail(P + E, 7);
}

// A few tokens on a handle with the single-kernel decode path: one single-token step per token,
// each streaming only its own experts (up to kDecodeLoopMaxT tokens).
bool decode_loop(const Dims &d, int T, bool want_counts) {
    return d.fast_decode && T >= 1 && (T == 1 || (T <= kDecodeLoopMaxT && !want_counts));
}

int decode_loop_max_tokens() { return kDecodeLoopMaxT; }

bool buckets_built(const Dims &d, int T, bool want_counts) {
    if (decode_loop(d, T, want_counts)) return false;
    return T > 1 || want_counts || (d.mma && d.mma_fmt);
}

cudaError_t launch_checks(const Params &p, int T, bool buckets, cudaStream_t st) {
    check_kernel<<<1, kThreads, 0, st>>>(p, T, buckets ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_forward(const Params &p0, const float *x, int T, float *y, cudaStream_t st,
                           bool want_buckets, cudaEvent_t *ev) {
    // this call's tensor-core work items: 128 tokens on the tcgen05 kernel (T >= kTcMinT),
    // else 32 on the mma.sync kernel
    Params p = p0;
    p.item_tok = mma_item_tokens(p0.d, T);
    const Dims &d = p.d;
    if (p.item_tok == kTcTok && !p.tmaps) return cudaErrorInvalidValue;   // the tcgen05 kernels read tensor maps
    if (T == 1 && d.fast_decode) return launch_decode_fast(p, x, y, st, ev, want_buckets);
    if (decode_loop(d, T, want_buckets)) {
        // token t: x, y and its top-K record at offset t (the steps run one after another on the
        // stream, each started early by the programmatic dependent launch)
        cudaError_t e = cudaSuccess;
        if (ev) e = cudaEventRecord(ev[0], st);
        if (e == cudaSuccess && ev) e = cudaEventRecord(ev[1], st);
        for (int t = 0; t < T && e == cudaSuccess; t++) {
            Params pt = p;
            pt.ws.topk_idx += (size_t)t * d.K;
            pt.ws.topk_w += (size_t)t * d.K;
            e = launch_decode_fast(pt, x + (size_t)t * d.H, y + (size_t)t * d.H, st, nullptr, false);
        }
        for (int i = 2; ev && e == cudaSuccess && i < 5; i++) e = cudaEventRecord(ev[i], st);
        return e;
    }
    const size_t smem = router_smem_bytes(d);
    const bool mma_all = d.mma && (T > 1 || d.mma_fmt);   // the tensor-core expert kernels
    const int buckets = buckets_built(d, T, want_buckets) ? 1 : 0;
    cudaError_t e = cudaSuccess;
    auto mark = [&](int i) {
        if (ev && e == cudaSuccess) e = cudaEventRecord(ev[i], st);
    };
    auto check = [&]() {
        if (e == cudaSuccess) e = cudaGetLastError();
    };
    mark(0);
    if (T <= kGemvMaxT) {
        const int grid = (d.E + 1) / 2;
        router_gemv_kernel<<<grid, kThreads, smem, st>>>(p, x, T, buckets);
    } else {
        const int S = router_split(T, d.E, d.H);
        const dim3 grid((d.E + kRtExp - 1) / kRtExp, (T + kRtTok - 1) / kRtTok, S);
        router_tiled_kernel<<<grid, kThreads, kRtSmem, st>>>(p, x, T);
        check();
        router_reduce_kernel<<<T, kThreads, smem, st>>>(p, x, T, S, buckets);
    }
    check();
    mark(1);
    if (T == 1 && !mma_all) {
        constexpr int RPW_GU = 2, RPW_D = 4;
        const dim3 g1((d.I_max + kWarps * RPW_GU - 1) / (kWarps * RPW_GU), d.K + d.n_shared);
        gateup_decode_kernel<RPW_GU><<<g1, kThreads, 0, st>>>(p);
        check();
        mark(2);
        const int g2 = (d.H + kWarps * RPW_D - 1) / (kWarps * RPW_D);
        down_decode_kernel<RPW_D><<<g2, kThreads, 0, st>>>(p, x, y);
        check();
        mark(3);
        mark(4);
        return e;
    }
    if (mma_all) {
        const int ni = max_items(T, d.K, d.E, d.n_shared, p.item_tok);
        const dim3 g1(ni, d.I_max / 128);
        launch_mma_phase<true>(p, T, g1, st);
        check();
        mark(2);
        const dim3 g2(ni, (d.H + 255) / 256);
        launch_mma_phase<false>(p, T, g2, st);
        check();
        mark(3);
        combine_kernel<<<dim3(T, (d.H + 4 * kThreads - 1) / (4 * kThreads)), kThreads, 0, st>>>(p, x, y, T);
        check();
        mark(4);
        return e;
    }
    constexpr int RPW_GU = 2, RPW_D = 4, NT = 4;
    const int slots = (d.E < T * d.K ? d.E : T * d.K) + d.n_shared;
    const dim3 g1((d.I_max + kWarps * RPW_GU - 1) / (kWarps * RPW_GU), slots);
    gateup_batched_kernel<RPW_GU, NT><<<g1, kThreads, 0, st>>>(p, T);
    check();
    mark(2);
    const dim3 g2((d.H + kWarps * RPW_D - 1) / (kWarps * RPW_D), slots);
    down_batched_kernel<RPW_D, NT><<<g2, kThreads, 0, st>>>(p, T);
    check();
    mark(3);
    combine_kernel<<<dim3(T, (d.H + 4 * kThreads - 1) / (4 * kThreads)), kThreads, 0, st>>>(p, x, y, T);
    check();
    mark(4);
    return e;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Router without any device allocation (moe_route_noalloc in moe.h).
//
// For callers that may not allocate device memory themselves: for example a
// host framework whose device memory all belongs to its own pool allocator,
// or a serving loop that must never call cudaMalloc/cudaFree because those
// calls can synchronise the device and can fail under memory pressure.  Such
// a caller cannot create a moe_handle (moe_init allocates the workspace), so
// this entry point takes the router weights and buffers directly and keeps
// its scratch (router logits and the last-block ticket) in one fixed static
// device array.  Every GPU that loads this library holds that array until
// the process exits.
// ---------------------------------------------------------------------------

#define MOE_NOALLOC_LOGITS (MOE_ROUTE_NOALLOC_MAX_TOKENS * MOE_ROUTE_NOALLOC_MAX_EXPERTS)

// [0, 64): ticket counter (and padding); [64, 64 + MOE_NOALLOC_LOGITS): logits
static __device__ __align__(256) float g_route_scratch[64 + MOE_NOALLOC_LOGITS];

namespace moe {
namespace {

__global__ void __launch_bounds__(kThreads) router_noalloc_kernel(Params p, const float *__restrict__ x,
                                                                  int T) {
    extern __shared__ float smem[];
    __shared__ float s_r[kGemvMaxT];
    const int H = p.d.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < T) {
        float ss = 0.0f;
        if (p.d.prenorm) {
            const float4 *x4 = reinterpret_cast<const float4 *>(x + (size_t)warp * H);
            for (int i = lane; i < H / 4; i += 32) {
                const float4 v = __ldg(x4 + i);
                ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
            }
            ss = warp_sum(ss);
        }
        if (lane == 0) s_r[warp] = p.d.prenorm ? 1.0f / sqrtf(ss / (float)H + p.d.eps) : 1.0f;
    }
    __syncthreads();
    gemv_logits(p, x, T, s_r);
    router_tail(p, T, 0, gridDim.x, smem);
}

constexpr int kMaxDevices = 64;

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const moe_config *cfg, const float *router_w,
                                        const float *router_bias, const float *x, int32_t T,
                                        int32_t *topk_idx, float *topk_w, void *stream) {
    using namespace moe;
    // Device address of the static scratch array, looked up once per device
    // with that device current (the host-side symbol is only a stand-in).
    static float *s_scratch[kMaxDevices] = {};
    static bool s_ready[kMaxDevices] = {};
    static std::mutex s_setup;
    if (!cfg || !router_w || !router_bias || !x || !topk_idx || !topk_w) return MOE_ERR_INVALID;
    if (cfg->hidden < 32 || cfg->hidden > 16384 || cfg->hidden % 32) return MOE_ERR_UNSUPPORTED;
    if (cfg->n_experts < 1 || cfg->n_experts > MOE_ROUTE_NOALLOC_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
    if (cfg->top_k < 1 || cfg->top_k > cfg->n_experts || cfg->top_k > 32) return MOE_ERR_INVALID;
    if (cfg->score_func != MOE_SCORE_SIGMOID && cfg->score_func != MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID;
    if (cfg->n_group < 1 || cfg->n_group > 32 || cfg->n_experts % cfg->n_group) return MOE_ERR_INVALID;
    if (cfg->n_group > 1 && (cfg->score_func != MOE_SCORE_SIGMOID || cfg->topk_group < 1 ||
                             cfg->topk_group > cfg->n_group ||
                             cfg->top_k > cfg->topk_group * (cfg->n_experts / cfg->n_group)))
        return MOE_ERR_INVALID;
    if (cfg->norm_topk != 0 && cfg->norm_topk != 1) return MOE_ERR_INVALID;
    if (T < 0 || T > MOE_ROUTE_NOALLOC_MAX_TOKENS) return MOE_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(router_w) | reinterpret_cast<uintptr_t>(x)) & 15u) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    Dims d = {};
    d.H = cfg->hidden;
    d.E = cfg->n_experts;
    d.ep_hi = d.E;
    d.K = cfg->top_k;
    d.norm_topk = cfg->norm_topk;
    d.n_group = cfg->n_group;
    d.topk_group = cfg->n_group > 1 ? cfg->topk_group : 1;
    d.score_func = cfg->score_func;
    d.prenorm = (cfg->flags & MOE_FLAG_PRENORM_RESIDUAL) ? 1 : 0;
    d.scale = cfg->routed_scale;
    d.eps = cfg->rms_eps;
    d.max_tokens = MOE_ROUTE_NOALLOC_MAX_TOKENS;
    const size_t smem = router_smem_bytes(d);
    std::unique_lock<std::mutex> lock(s_setup);
    if (!s_ready[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_route_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
        const int max_smem = (int)((size_t)kWarps * 2 * MOE_ROUTE_NOALLOC_MAX_EXPERTS * sizeof(float));
        if (cudaFuncSetAttribute(router_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 max_smem) != cudaSuccess)
            return MOE_ERR_CUDA;
        s_scratch[dev] = static_cast<float *>(ptr);
        s_ready[dev] = true;
    }
    float *scratch = s_scratch[dev];
    lock.unlock();
    Params p = {};
    p.d = d;
    p.router_w = router_w;
    p.router_b = router_bias;
    p.ws.counters = reinterpret_cast<unsigned *>(scratch);
    p.ws.logits = scratch + 64;
    p.ws.topk_idx = topk_idx;
    p.ws.topk_w = topk_w;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The ticket must start at zero; logits are fully rewritten by every call.
    if (cudaMemsetAsync(p.ws.counters, 0, sizeof(unsigned), st) != cudaSuccess) return MOE_ERR_CUDA;
    const int grid = (d.E + 1) / 2;
    router_noalloc_kernel<<<grid, kThreads, smem, st>>>(p, x, T);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
