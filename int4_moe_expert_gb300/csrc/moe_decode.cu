// Decode (T == 1): the whole MoE step as one persistent kernel.
//
// One block per SM (all resident together: one block fills an SM), eight
// warps.  The step's four parts run as phases separated by grid-wide
// barriers:
//   phase 0  one batch of loads (x chunk and this block's two router rows);
//            router logits -> sigmoid and selection score (sigmoid + bias);
//            (thread 0 arrives at barrier 1 once the scores are out); x digits
//            (a warp whose first unit is the shared expert's starts its loads
//            once the router rows are in)
//   routing  warp 0 of every block selects the top K (K rounds of a warp max)
//   phase 1  gate/up + SwiGLU: warp gw computes units gw, gw + nw, ... (nw =
//            warps in the grid); a unit is the (gate row, up row) pair of one
//            output, the shared expert's units first, then slot by slot
//            (each warp then starts loading its first down unit) -> barrier 2
//   phase 2  down: each half-block (4 warps) serves one slot, quantises that
//            slot's h once into shared memory, and its warps take units of
//            four output rows; d_j = w_j * s_d * (Q_d h_j)          -> barrier 3
//   phase 3  y = sum_k d_k + d_shared (k ascending; + x with pre-norm residual)
//
// What is computed (reader.mx "25GB 内存上运行 GLM 5.2 744B" section 11;
// devpress GLM-5.2 breakdown "Step 6 (MoE)" 6a-6d; Edge0 article section 七):
// l = W_r x, sigma = sigmoid(l), top-K of sigma + bias (lower index wins a
// tie), w = s sigma / (sum sigma + 1e-20); g = s_g (Q_g x), u = s_u (Q_u x),
// h = silu(g) u, d = s_d (Q_d h), y = sum_k w_k d_k + d_shared.
//
// Arithmetic.  An activation vector v (x, or one expert's h) is held as
// 16-bit fixed point with one scale per vector: X_i = rint(v_i / s),
// s = max|v| / 32639, |X_i| <= 32639 = 0x7F7F, written as two signed base-256
// digits X = d1 256 + d0, each in [-128, 127] (kPlanes; three planes give
// 24-bit fixed point).  A packed int4 weight byte holds two unsigned nibbles
// n = q + 8 (section 06 format), so one row's dot product is
//     sum_i q_i v_i = s * sum_p 256^p (sum_i n_i d_{p,i} - 8 sum_i d_{p,i}),
// with every inner sum exact in int32 (dp4a: four unsigned nibble bytes times
// four signed digit bytes).  Only the final plane combination and the scale
// are floating point.  The representation error of v is at most
// max|v| * 2^-16 per element (measured against a double-precision evaluation: 1.1e-4
// worst relative error on the GLM layer, 5e-4 after 40 chained layers).
//
// Digits in shared memory: for chunk c (elements 32c..32c+31, one 16-byte
// weight load) and q = 2p + lh (q < kQ), the uint4 at [q * C + c] holds, in word m,
// the plane-p digits of elements 8m+{0,2,4,6} (lh = 0: the low nibbles of
// word m) or 8m+{1,3,5,7} (lh = 1: the high nibbles), one per byte.
//
// Weights go straight from HBM into registers with 16-byte non-caching loads:
// lane l holds chunks l, l + 32, ... of every row of its unit, which is the
// layout the dp4a loop reads, and the next unit's loads are in flight while
// the current one is computed.  (Measured on this GPU, streaming 105 MB with
// 8 warps per SM: per-warp units loaded into registers ran at 5.8 TB/s, the
// same units through cp.async or 1-D bulk copies into shared memory at
// 5.0-5.1 TB/s, with or without compute.)
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDnRows = 4;          // output rows per down unit
constexpr int kSmemBudget = 64 * 1024;
constexpr unsigned long long kWaitNs = 500ull * 1000 * 1000;   // every wait gives up after 0.5 s
constexpr int kPlanes = 2;                  // activation digits (bytes of fixed point) per value
constexpr int kQ = 2 * kPlanes;             // digit words (uint4) per 32-value chunk
constexpr int kQMaxInt = kPlanes == 2 ? 0x7F7F : 0x7F7F7F;   // largest |X| with balanced digits
constexpr unsigned kBias = kPlanes == 2 ? 0x8080u : 0x808080u;
constexpr float kQMax = (float)kQMaxInt;
constexpr int kSwWords = (kMaxSlots + 3) / 4 * 4;   // s_w padded to 16 bytes
constexpr int kPtab = 4;       // expert pointers each thread stages: E <= kPtab * kThreads
constexpr int kKeyBatch = 8;   // score loads a routing lane has in flight at once
static_assert(kMaxSlots * 16 % 16 == 0 && kSwWords >= kMaxSlots, "shared-memory carving");
static_assert(kPtab * kThreads >= 1024, "pointer staging covers the largest expert count");

enum : unsigned { kErrGrid = MOE_DEVICE_ERR_GRID };

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void dp4a_us(int &acc, uint32_t nib, uint32_t dig) {
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(nib), "r"(dig));
}

__device__ __forceinline__ void dp4a_ss(int &acc, uint32_t w, uint32_t dig) {
    asm("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(w), "r"(dig));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int m) {
    return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// (s, b) of an int4 affine group (float16 pair, s in the low half of the word)
__device__ __forceinline__ float g64_s(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float g64_b(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

__device__ __forceinline__ float planes_lh_to_float(const int (&lo)[kPlanes], const int (&hi)[kPlanes]) {
    float r = 0.0f;
#pragma unroll
    for (int p = kPlanes - 1; p >= 0; p--) r = fmaf(r, 256.0f, __int2float_rn(lo[p] + (hi[p] >> 4)));
    return r;
}

// Digits of the 32 values of one chunk (natural order) scaled by inv = 1/s;
// dsum[p] = sum of the plane-p digits.  With U = X + kBias (>= 0), byte p of U
// minus 128 is the balanced digit d_p, i.e. byte p of U xor 0x80 read as a
// signed byte; bytes are gathered into words with byte permutes.
__device__ __forceinline__ void quant_chunk(const float (&v)[32], float inv, uint4 (&dig)[kQ], int (&dsum)[kPlanes]) {
    uint32_t U[32];
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const int X = min(max(__float2int_rn(v[i] * inv), -kQMaxInt), kQMaxInt);
        U[i] = (uint32_t)(X + (int)kBias);
    }
    uint32_t w[kQ][4];
#pragma unroll
    for (int m = 0; m < 4; m++) {
#pragma unroll
        for (int lh = 0; lh < 2; lh++) {
            const int e0 = 8 * m + lh;       // elements e0, e0 + 2, e0 + 4, e0 + 6
#pragma unroll
            for (int p = 0; p < kPlanes; p++) {
                const uint32_t sel = (uint32_t)p | ((uint32_t)(4 + p) << 4);
                const uint32_t a = __byte_perm(U[e0], U[e0 + 2], sel);
                const uint32_t b = __byte_perm(U[e0 + 4], U[e0 + 6], sel);
                w[2 * p + lh][m] = __byte_perm(a, b, 0x5410) ^ 0x80808080u;
            }
        }
    }
#pragma unroll
    for (int q = 0; q < kQ; q++) dig[q] = make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
#pragma unroll
    for (int p = 0; p < kPlanes; p++) {
        int t = 0;
#pragma unroll
        for (int m = 0; m < 4; m++) {
            t = __dp4a((int)w[2 * p][m], 0x01010101, t);
            t = __dp4a((int)w[2 * p + 1][m], 0x01010101, t);
        }
        dsum[p] = t;
    }
}

// lo[rr][p] += low-nibble sums, hi[rr][p] += 16 x high-nibble sums for NR
// rows of one chunk, issued so that consecutive dp4a go to different rows.
template <int NR>
__device__ __forceinline__ void dot_rows(const uint4 (&w)[NR], const uint4 (&dig)[kQ], int (&lo)[NR][kPlanes],
                                         int (&hi)[NR][kPlanes]) {
#pragma unroll
    for (int m = 0; m < 4; m++) {
        uint32_t l[NR], h[NR];
#pragma unroll
        for (int rr = 0; rr < NR; rr++) {
            const uint32_t word = word_of(w[rr], m);
            l[rr] = word & 0x0F0F0F0Fu;
            h[rr] = word & 0xF0F0F0F0u;
        }
#pragma unroll
        for (int p = 0; p < kPlanes; p++) {
            const uint32_t dl = word_of(dig[2 * p], m), dh = word_of(dig[2 * p + 1], m);
#pragma unroll
            for (int rr = 0; rr < NR; rr++) dp4a_us(lo[rr][p], l[rr], dl);
#pragma unroll
            for (int rr = 0; rr < NR; rr++) dp4a_us(hi[rr][p], h[rr], dh);
        }
    }
}

// int8 rows (one signed byte per weight, natural order): lo[rr][p] += the plane-p sums of NR
// rows of one 32-value chunk (w[rr][0..1]: the chunk's 32 bytes).  The digit words hold the
// even and the odd elements of 8 consecutive values apart (the int4 nibble order above); a
// byte permute puts the digits of elements 4 jw .. 4 jw + 3 in order again.
template <int NR>
__device__ __forceinline__ void dot8_rows(const uint4 (&w)[NR][2], const uint4 (&dig)[kQ], int (&lo)[NR][kPlanes]) {
#pragma unroll
    for (int jw = 0; jw < 8; jw++) {
#pragma unroll
        for (int p = 0; p < kPlanes; p++) {
            const uint32_t de = word_of(dig[2 * p], jw >> 1), dd = word_of(dig[2 * p + 1], jw >> 1);
            const uint32_t dn = __byte_perm(de, dd, (jw & 1) ? 0x7362 : 0x5140);
#pragma unroll
            for (int rr = 0; rr < NR; rr++) dp4a_ss(lo[rr][p], word_of(w[rr][jw >> 2], jw & 3), dn);
        }
    }
}

// Reduce NV floats per lane over the warp so that lane l ends holding the
// total of value l / (32 / NV) (NV = 2, 4, 8 or 16): a reduce-scatter
// butterfly, the same fixed order on every call.
template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane) {
#pragma unroll
    for (int o = 16, n = NV; n > 1; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; i++) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = 32 / NV / 2; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

// Unsigned key with the order of the float (no NaN; -0 not used); every
// float, -inf included, maps above 0, which marks a removed entry.
__device__ __forceinline__ unsigned order_key(float f) {
    const unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Single thread: wait until *ctr has reached target (counters only grow;
// wrap-safe).  false if the wait ran out (kWaitNs).
__device__ bool spin_until(const unsigned *ctr, unsigned target) {
    const unsigned long long t0 = now_ns();
    for (;;) {
        for (int i = 0; i < 32; i++) {
            if ((int)(ld_acquire(ctr) - target) >= 0) return true;
            __nanosleep(32);
        }
        if (now_ns() - t0 > kWaitNs) return false;
    }
}
// Whole block: every block adds one to *ctr, then waits for all of them.
__device__ bool grid_barrier(unsigned *ctr, unsigned target, unsigned *err, volatile int *s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        const bool ok = spin_until(ctr, target);
        if (!ok) atomicOr(err, kErrGrid);
        *s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    return *s_ok != 0;
}


struct FusedShape {
    // gate/up: a unit is one (gate row, up row) pair of one slot
    int C;             // chunks per row = H / 32
    int rowbytes;      // H / 2
    int U_sh, U_r;     // units of the shared expert, units per routed expert
    int gu_units;
    // down: a unit is kDnRows consecutive output rows of one slot
    int Cd;            // chunks per row = I / 32
    int drowbytes;     // I / 2
    int J;             // slots = K + n_shared
    int RB;            // row blocks = H / kDnRows
    int dig_bytes;     // digits: x (7 C uint4) in phases 0/1, two slots' h (2 x 7 Cd uint4) in phase 2
    size_t smem;
};

__host__ __device__ inline FusedShape fused_shape(const Dims &d) {
    FusedShape s;
    s.C = d.H / 32;
    s.rowbytes = d.H / 2;
    s.U_sh = d.n_shared ? d.I_sh : 0;
    s.U_r = d.I;
    s.gu_units = s.U_sh + d.K * s.U_r;
    s.Cd = d.I / 32;
    s.drowbytes = d.I / 2;
    s.J = d.K + d.n_shared;
    s.RB = d.H / kDnRows;
    s.dig_bytes = (kQ + 1) * 16 * (s.C > 2 * s.Cd ? s.C : 2 * s.Cd);
    // digits | red[64] | slab[33] | scale[33] | w[36] | flags[4] | score keys[E] | sel[32] | sigmoids[E]
    // | expert slab pointers[E] | expert scale pointers[E]   (E padded to 4 entries)
    const size_t e4 = (size_t)(d.E + 3) / 4 * 4;
    s.smem = (size_t)s.dig_bytes + 64 * 4 + kMaxSlots * 16 + kSwWords * 4 + 16 + e4 * 4 + 32 * 4 + e4 * 4 + e4 * 16;
    return s;
}

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {   // weights: read once, keep out of L1
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Routing variants, warp 0 of a block (all E scores written): s_sig[e] = the expert's gate
// value (sigmoid, or the softmax probability), s_key[e] = the order key of its selection
// score, 0 never (a removed entry); each lane's best key among experts lane + 32 i.
//   softmax family: g = exp(l - max l) / sum exp(l - max l), selection by g;
//   group-limited sigmoid: a group's score is the sum of its two best (sigma + bias),
//   the topk_group best groups are kept (a tie to the lower group) and the others'
//   experts rank below every kept one (score -inf).
__device__ __forceinline__ void route_variant_keys(const Params &p, int E, int lane, unsigned *s_key,
                                                float *s_sig, unsigned &best, int &bidx) {
    const unsigned kFull = 0xffffffffu;
    const bool softmax = p.d.score_func == MOE_SCORE_SOFTMAX;
    float *s_ch = reinterpret_cast<float *>(s_key);    // choices as floats until the keys replace them
    float lmax = -INFINITY;
    for (int e0 = lane; e0 < E; e0 += 32 * kKeyBatch) {
        float c[kKeyBatch], sgv[kKeyBatch];
#pragma unroll
        for (int i = 0; i < kKeyBatch; i++) {
            const int e = e0 + 32 * i;
            c[i] = e < E ? __ldcg(p.ws.dscore + E + e) : 0.0f;
            sgv[i] = (e < E && !softmax) ? __ldcg(p.ws.dscore + e) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < kKeyBatch; i++) {
            const int e = e0 + 32 * i;
            if (e < E) {
                s_ch[e] = c[i];
                s_sig[e] = sgv[i];
                lmax = fmaxf(lmax, c[i]);
            }
        }
    }
    if (softmax) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(kFull, lmax, o));
        float z = 0.0f;
        for (int e = lane; e < E; e += 32) {
            const float v = expf(s_ch[e] - lmax);
            s_sig[e] = v;
            z += v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(kFull, z, o);
        for (int e = lane; e < E; e += 32) {
            const float g = s_sig[e] / z;
            s_sig[e] = g;
            s_ch[e] = isnan(g) ? -INFINITY : g;
        }
    }
    __syncwarp();
    if (p.d.n_group > 1) {
        const int G = p.d.n_group, m = E / G;
        float gsc = -INFINITY;
        if (lane < G) {
            float b1 = -INFINITY, b2 = -INFINITY;
            for (int i = 0; i < m; i++) {
                const float v = s_ch[lane * m + i];
                if (v > b1) { b2 = b1; b1 = v; }
                else if (v > b2) b2 = v;
            }
            gsc = m > 1 ? b1 + b2 : b1;
        }
        unsigned keep = 0u;
        bool taken = false;
        for (int r = 0; r < p.d.topk_group; r++) {
            const unsigned k = (lane < G && !taken) ? order_key(gsc) : 0u;
            const unsigned mx = __reduce_max_sync(kFull, k);
            const unsigned g = __reduce_min_sync(kFull, (k == mx && lane < G && !taken) ? (unsigned)lane : 0xffffffffu);
            keep |= 1u << g;
            if (lane == (int)g) taken = true;
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32)
            if (!((keep >> (e / m)) & 1u)) s_ch[e] = -INFINITY;
        __syncwarp();
    }
    for (int e = lane; e < E; e += 32) {
        const unsigned k = order_key(s_ch[e]);
        s_key[e] = k;
        if (k > best) { best = k; bidx = e; }
    }
    __syncwarp();
}

// V = 0: the sigmoid + bias router with plain top-K (GLM-5.2, n_group == 1), int4 experts.
// V = 1: the routing variants (Edge0 article section 七; reader.mx section 03): group-limited
// selection (n_group > 1, sigmoid family) and the softmax family; only warp 0's selection
// differs.  V = 2: any of those routers, and int8 routed and/or shared experts (reader.mx
// section 03, the OLMoE engine; section 06/07, the GLM engine's int8 shared expert): an int8
// unit's rows are twice as long, so it is streamed in two column segments of about half the
// chunks each (the same registers as an int4 unit), its partial sums carried between them.
template <int CPLH, int CPLI, int V>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(Params p, const float *__restrict__ x,
                                                                   float *__restrict__ y, FusedShape sh,
                                                                   int want_counts) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint4 *xdig = reinterpret_cast<uint4 *>(smem);
    int4 *xdsum = reinterpret_cast<int4 *>(xdig + kQ * sh.C);
    float *red = reinterpret_cast<float *>(smem + sh.dig_bytes);
    const uint8_t **s_slab = reinterpret_cast<const uint8_t **>(red + 64);
    const float **s_scale = reinterpret_cast<const float **>(s_slab + kMaxSlots);
    float *s_w = reinterpret_cast<float *>(s_scale + kMaxSlots);
    volatile int *s_flags = reinterpret_cast<volatile int *>(s_w + kSwWords);   // [0] ok [1] abort
    unsigned *s_key = reinterpret_cast<unsigned *>(const_cast<int *>(s_flags + 4));   // [E] (+pad)
    int *s_sel = reinterpret_cast<int *>(s_key + (p.d.E + 3) / 4 * 4);                // [32]
    float *s_sig = reinterpret_cast<float *>(s_sel + 32);                               // [E] (+pad)
    const uint8_t **s_pslab = reinterpret_cast<const uint8_t **>(s_sig + (p.d.E + 3) / 4 * 4);   // [E] (+pad)
    const float **s_pscale = reinterpret_cast<const float **>(s_pslab + (p.d.E + 3) / 4 * 4);    // [E] (+pad)

    const Dims &d = p.d;
    const int H = d.H, E = d.E, K = d.K, J = sh.J, C = sh.C, Cd = sh.Cd;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int G = gridDim.x, nw = G * kWarps, gw = blockIdx.x * kWarps + warp;
    const unsigned kFull = 0xffffffffu;
    unsigned *bar1 = p.ws.counters + 4, *bar2 = p.ws.counters + 5, *bar3 = p.ws.counters + 6;
    unsigned *epoch = p.ws.counters + 7;
    const bool fullH = (C % 32) == 0, fullI = (Cd % 32) == 0;
    // timeline (MOE_FLAG_TRACE): block b's record of MOE_TRACE_SLOTS global-timer readings
    const bool trace = p.d.trace != 0 && blockIdx.x < kTraceBlocks;
    unsigned long long *tr = p.ws.trace + (size_t)blockIdx.x * MOE_TRACE_SLOTS;
    auto mark = [&](int slot) {
        if (trace && tid == 0) tr[slot] = now_ns();
    };

    // ---- gate/up units: unit u < U_sh is row u of the shared expert, unit U_sh + v is row
    // v mod I of slot v / I.  The shared expert's units go to warps 1..7 (their share
    // sw = 7 block + warp - 1, sw + nsw, ... with nsw = 7 G), since warp 0 spends that time
    // routing; then every warp takes routed units U_sh + gw, U_sh + gw + nw, ...  A unit's
    // rows go straight into registers (lane l: chunks l + 32 k of the gate row, then of
    // the up row); the next unit's loads are in flight while the current one is computed.
    // A unit is held as (pos, o): pos -1 the shared expert, 0..K-1 a routed slot; o its row.
    // Units are stepped incrementally (no division per unit).
    struct Unit { int pos, o; };
    const int nsw = 7 * G, sw = 7 * blockIdx.x + warp - 1;
    const Unit r_first = {gw / d.I, gw % d.I};       // routed unit U_sh + gw
    const Unit u_first = (warp > 0 && sw < sh.U_sh) ? Unit{-1, sw} : r_first;
    auto next_unit = [&](Unit u) -> Unit {
        if (u.pos < 0) {
            const int n = u.o + nsw;
            return n < sh.U_sh ? Unit{-1, n} : r_first;
        }
        int pos = u.pos, o = u.o + nw;
        while (o >= d.I) { o -= d.I; pos++; }
        return Unit{pos, o};
    };
    auto load_gu = [&](Unit u, uint4 (&w)[2 * CPLH], float &sg, float &su) {
        const int o = u.o;
        const int Ij = u.pos < 0 ? d.I_sh : d.I;
        const uint8_t *slab = u.pos < 0 ? p.sh_slab : s_slab[u.pos];
        const float *scale = u.pos < 0 ? p.sh_scale : s_scale[u.pos];
        const uint4 *g = reinterpret_cast<const uint4 *>(slab + (size_t)o * sh.rowbytes) + lane;
        const uint4 *up = reinterpret_cast<const uint4 *>(slab + (size_t)(Ij + o) * sh.rowbytes) + lane;
#pragma unroll
        for (int k = 0; k < CPLH; k++) {
            if (fullH || lane + 32 * k < C) {
                w[k] = ldg_stream(g + 32 * k);
                w[CPLH + k] = ldg_stream(up + 32 * k);
            }
        }
        if (lane == 0) {
            sg = __ldg(scale + o);
            su = __ldg(scale + Ij + o);
        }
    };
    // V == 2: a gate/up step is one segment of a unit (int4 units: one segment, the whole rows;
    // int8 units: two, chunks [0, SEG) and [SEG, CPLH) of each row, 2 uint4 per chunk)
    constexpr int SEG = (CPLH + 1) / 2;
    constexpr int NBUF = V == 2 ? 2 * (CPLH > 2 * SEG ? CPLH : 2 * SEG) : 2 * CPLH;
    const bool r8 = V == 2 && d.expert_fmt == MOE_FORMAT_INT8;
    const bool s8 = V == 2 && d.shared_fmt == MOE_FORMAT_INT8;
    // V == 2, int4 affine group-64 (Edge0 article section 三): int4 rows of unsigned nibbles u and
    // one (s, b) pair per 64 inputs; a chunk (32 inputs) contributes s sum(u X) + b sum(X)
    const bool rg = V == 2 && d.expert_fmt == MOE_FORMAT_G64;
    const bool sgf = V == 2 && d.shared_fmt == MOE_FORMAT_G64;
    auto isg = [&](const Unit &u) { return u.pos < 0 ? sgf : rg; };
    struct Step { Unit u; int seg; };
    auto is8 = [&](const Unit &u) { return u.pos < 0 ? s8 : r8; };
    auto next_step = [&](Step st) -> Step {
        if (is8(st.u) && st.seg == 0) return Step{st.u, 1};
        return Step{next_unit(st.u), 0};
    };
    auto load_step = [&](Step st, uint4 (&w)[NBUF], float &sg, float &su, uint32_t (&pr)[2 * CPLH]) {
        const int o = st.u.o;
        const int Ij = st.u.pos < 0 ? d.I_sh : d.I;
        const uint8_t *slab = st.u.pos < 0 ? p.sh_slab : s_slab[st.u.pos];
        const float *scale = st.u.pos < 0 ? p.sh_scale : s_scale[st.u.pos];
        if (!is8(st.u)) {
            const uint4 *g = reinterpret_cast<const uint4 *>(slab + (size_t)o * sh.rowbytes) + lane;
            const uint4 *up = reinterpret_cast<const uint4 *>(slab + (size_t)(Ij + o) * sh.rowbytes) + lane;
#pragma unroll
            for (int k = 0; k < CPLH; k++) {
                if (fullH || lane + 32 * k < C) {
                    w[k] = ldg_stream(g + 32 * k);
                    w[NBUF / 2 + k] = ldg_stream(up + 32 * k);
                }
            }
        } else {                          // int8 rows: H bytes, chunk c at bytes 32 c .. 32 c + 31
            const uint4 *g = reinterpret_cast<const uint4 *>(slab + (size_t)o * H);
            const uint4 *up = reinterpret_cast<const uint4 *>(slab + (size_t)(Ij + o) * H);
#pragma unroll
            for (int t = 0; t < SEG; t++) {
                const int k = st.seg * SEG + t, c = lane + 32 * k;
                if (k < CPLH && (fullH || c < C)) {
                    w[2 * t] = ldg_stream(g + 2 * c);
                    w[2 * t + 1] = ldg_stream(g + 2 * c + 1);
                    w[NBUF / 2 + 2 * t] = ldg_stream(up + 2 * c);
                    w[NBUF / 2 + 2 * t + 1] = ldg_stream(up + 2 * c + 1);
                }
            }
        }
        if (isg(st.u)) {                  // the chunks' (s, b) pairs; no per-row scale
            const uint32_t *pw = reinterpret_cast<const uint32_t *>(scale);
            const int ng = H / 64;
#pragma unroll
            for (int k = 0; k < CPLH; k++) {
                const int c = lane + 32 * k;
                if (fullH || c < C) {
                    pr[k] = __ldg(pw + (size_t)o * ng + (c >> 1));
                    pr[CPLH + k] = __ldg(pw + (size_t)(Ij + o) * ng + (c >> 1));
                }
            }
        } else if (lane == 0) {
            sg = __ldg(scale + o);
            su = __ldg(scale + Ij + o);
        }
    };
    uint32_t pra[2 * CPLH], prb[2 * CPLH];   // V == 2, group-64 units: (s, b) pairs of the buffered unit
    uint4 wa[NBUF], wb[NBUF];
    float sga = 0.0f, sua = 0.0f, sgb = 0.0f, sub = 0.0f;
    bool loaded = false;          // wa holds the warp's first unit

    // ---- phase 0: one batch of loads: x chunk `tid`, the same chunk of this block's two router rows
    // (issued before the shared-expert prefetch: routing is on the critical path)
    const int e0 = 2 * blockIdx.x;
    const bool has0 = e0 < E, has1 = e0 + 1 < E;
    float xv[32];
    float a0 = 0.0f, a1 = 0.0f, amax = 0.0f, ss = 0.0f;
    bool bad = false;
    float4 u0[8], u1[8];
    float bias0 = 0.0f, bias1 = 0.0f;
    if (tid == 0) {
        if (has0) bias0 = __ldg(p.router_b + e0);
        if (has1) bias1 = __ldg(p.router_b + e0 + 1);
    }
    // Before the wait for the preceding grid (programmatic dependent launch): only reads of
    // data no call writes -- this block's chunk of its two router rows, the biases and every
    // expert's slab and scale pointers (for the slot tables after routing; E <= 4 x kThreads).
    // These overlap the previous kernel's tail when calls follow one another on a stream.
    // (A shared-expert warp's first unit is requested only once the router rows are in:
    // issued together, the two compete for HBM and routing, the critical path, starts later;
    // measured on the GLM-5.2 layer back to back, 40.2 -> 39.9 us per call with the early
    // barrier arrival below.)
    if (tid < C) {
        const float4 *w0 = reinterpret_cast<const float4 *>(p.router_w + (size_t)(has0 ? e0 : 0) * H + (size_t)tid * 32);
        const float4 *w1 = reinterpret_cast<const float4 *>(p.router_w + (size_t)(has1 ? e0 + 1 : 0) * H + (size_t)tid * 32);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            u0[k] = has0 ? __ldg(w0 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
            u1[k] = has1 ? __ldg(w1 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    const uint8_t *pt_slab[kPtab];
    const float *pt_scale[kPtab];
#pragma unroll
    for (int i = 0; i < kPtab; i++) {
        const int e = tid + i * kThreads;
        pt_slab[i] = e < E ? p.slabs[e] : nullptr;
        pt_scale[i] = e < E ? p.scales[e] : nullptr;
    }
    // x (possibly the previous call's output) and the handle's workspace (the previous call on
    // this handle uses it) only after the preceding grid has completed and its writes are
    // visible; the next call may then be launched (its blocks start as these exit)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // this call's number on the handle: the previous call's + 1, kept in device memory (so a
    // captured graph replays correctly); block 0 advances it once every block is past
    // barrier 2, i.e. after every block has read it.  Only thread 0 uses it.
    const unsigned gen = tid == 0 ? *reinterpret_cast<volatile unsigned *>(epoch) + 1u : 0u;
    const unsigned target = gen * (unsigned)G;
    if (trace && tid < MOE_TRACE_SLOTS) tr[tid] = 0ull;
    mark(0);
    if (tid == 0) s_flags[2] = 0;     // routing not known yet (read after the first __syncthreads)
    if (tid < C) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x + (size_t)tid * 32);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const float4 f = __ldg(x4 + k);
            xv[4 * k] = f.x; xv[4 * k + 1] = f.y; xv[4 * k + 2] = f.z; xv[4 * k + 3] = f.w;
        }
    }
    if (tid < C) {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            a0 = fmaf(u0[k].x, xv[4 * k], fmaf(u0[k].y, xv[4 * k + 1], fmaf(u0[k].z, xv[4 * k + 2], fmaf(u0[k].w, xv[4 * k + 3], a0))));
            a1 = fmaf(u1[k].x, xv[4 * k], fmaf(u1[k].y, xv[4 * k + 1], fmaf(u1[k].z, xv[4 * k + 2], fmaf(u1[k].w, xv[4 * k + 3], a1))));
        }
#pragma unroll
        for (int i = 0; i < 32; i++) {
            amax = fmaxf(amax, fabsf(xv[i]));
            ss = fmaf(xv[i], xv[i], ss);
            bad |= !isfinite(xv[i]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        ss += __shfl_xor_sync(kFull, ss, o);
        a0 += __shfl_xor_sync(kFull, a0, o);
        a1 += __shfl_xor_sync(kFull, a1, o);
    }
    bad = __any_sync(kFull, bad);
    if (lane == 0) {
        red[warp] = amax;
        red[8 + warp] = ss;
        red[16 + warp] = bad ? 1.0f : 0.0f;
        red[24 + warp] = a0;
        red[32 + warp] = a1;
    }
    __syncthreads();
    if (u_first.pos < 0) {
        if constexpr (V == 2) load_step(Step{u_first, 0}, wa, sga, sua, pra);
        else load_gu(u_first, wa, sga, sua);
        loaded = true;
    }
    amax = 0.0f;
    ss = 0.0f;
    bad = false;
    float A0 = 0.0f, A1 = 0.0f;
    for (int w = 0; w < kWarps; w++) {
        amax = fmaxf(amax, red[w]);
        ss += red[8 + w];
        bad |= red[16 + w] != 0.0f;
        A0 += red[24 + w];
        A1 += red[32 + w];
    }
    const float r = d.prenorm ? 1.0f / sqrtf(ss / (float)H + d.eps) : 1.0f;
    auto put_score = [&](int e, float raw, float bias) {
        const float l = raw * r;
        if constexpr (V != 0) {
            if (d.score_func == MOE_SCORE_SOFTMAX) {   // the routing warps take the softmax
                p.ws.logits[e] = l;
                p.ws.dscore[E + e] = l;
                return;
            }
        }
        const float sg = 1.0f / (1.0f + expf(-l));
        float c = sg + bias + 0.0f;   // + 0: no negative zero
        if (isnan(c)) c = -INFINITY;
        p.ws.logits[e] = l;
        p.ws.dscore[e] = sg;
        p.ws.dscore[E + e] = c;
    };
    if (tid == 0) {
        if (has0) put_score(e0, A0, bias0);
        if (has1) put_score(e0 + 1, A1, bias1);
    }
    // more experts than 2 per block: further pairs, rows split over all threads
    for (int ep = e0 + 2 * G; ep < E; ep += 2 * G) {
        const bool h1 = ep + 1 < E;
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        const float4 *w0 = reinterpret_cast<const float4 *>(p.router_w + (size_t)ep * H);
        const float4 *w1 = reinterpret_cast<const float4 *>(p.router_w + (size_t)(h1 ? ep + 1 : ep) * H);
        float b0 = 0.0f, b1 = 0.0f;
        for (int i = tid; i < H / 4; i += kThreads) {
            const float4 xq = __ldg(x4 + i), v0 = __ldg(w0 + i), v1 = __ldg(w1 + i);
            b0 = fmaf(v0.x, xq.x, fmaf(v0.y, xq.y, fmaf(v0.z, xq.z, fmaf(v0.w, xq.w, b0))));
            b1 = fmaf(v1.x, xq.x, fmaf(v1.y, xq.y, fmaf(v1.z, xq.z, fmaf(v1.w, xq.w, b1))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            b0 += __shfl_xor_sync(0xffffffffu, b0, o);
            b1 += __shfl_xor_sync(0xffffffffu, b1, o);
        }
        __syncthreads();
        if (lane == 0) { red[40 + warp] = b0; red[48 + warp] = b1; }
        __syncthreads();
        if (tid == 0) {
            float B0 = 0.0f, B1 = 0.0f;
            for (int w = 0; w < kWarps; w++) { B0 += red[40 + w]; B1 += red[48 + w]; }
            put_score(ep, B0, __ldg(p.router_b + ep));
            if (h1) put_score(ep + 1, B1, __ldg(p.router_b + ep + 1));
        }
    }

    // arrive at barrier 1 as soon as this block's scores are out (thread 0 wrote all of them),
    // not after the x digits: every block's arrival is on the routing critical path
    if (tid == 0) {
        __threadfence();
        atomicAdd(bar1, 1u);
    }
#pragma unroll
    for (int i = 0; i < kPtab; i++) {
        const int e = tid + i * kThreads;
        if (e < E) {
            s_pslab[e] = pt_slab[i];
            s_pscale[e] = pt_scale[i];
        }
    }

    // x digits (pre-normed when asked), from the registers already loaded
    const float m = amax * r;
    const float s_x = bad ? __int_as_float(0x7fc00000) : m / kQMax;
    const float inv = (m > 0.0f && !bad) ? kQMax / m : 0.0f;
    if (tid < C) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; i++) v[i] = xv[i] * r;
        uint4 dig[kQ];
        int ds[kPlanes];
        quant_chunk(v, inv, dig, ds);
#pragma unroll
        for (int q = 0; q < kQ; q++) xdig[q * C + tid] = dig[q];
        xdsum[tid] = make_int4(ds[0], ds[1], kPlanes > 2 ? ds[kPlanes - 1] : 0, 0);
    }

    // ---- barrier 1 and routing: warp 0 waits for every block's scores and picks the top K
    // while warps 1..7 compute the shared expert's units (those need no routing);
    // s_flags[2] then tells the block: 1 routing known (slot tables written), 2 failed
    mark(1);
    __syncthreads();              // this block's scores and x digits are written
    if (warp == 0) {
        bool ok = true;
        if (lane == 0) {
            ok = spin_until(bar1, target);
            if (!ok) atomicOr(p.ws.err, kErrGrid);
        }
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (!ok) {
            if (lane == 0) s_flags[2] = 2;
            return;
        }
        if (trace && lane == 0) tr[7] = now_ns();
        // top K by (score desc, index asc): K rounds of a warp-wide max over each
        // lane's best remaining expert (lane l holds experts l + 32 i)
        // (the scores of up to kKeyBatch x 32 experts are requested together: one round trip)
        unsigned best = 0u;
        int bidx = 0x7fffffff;
        if constexpr (V != 0) {
            route_variant_keys(p, E, lane, s_key, s_sig, best, bidx);
        } else
        for (int e0 = lane; e0 < E; e0 += 32 * kKeyBatch) {
            float c[kKeyBatch], sgv[kKeyBatch];
#pragma unroll
            for (int i = 0; i < kKeyBatch; i++) {
                const int e = e0 + 32 * i;
                c[i] = e < E ? __ldcg(p.ws.dscore + E + e) : 0.0f;
                sgv[i] = e < E ? __ldcg(p.ws.dscore + e) : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < kKeyBatch; i++) {
                const int e = e0 + 32 * i;
                if (e < E) {
                    const unsigned k = order_key(c[i]);
                    s_key[e] = k;
                    s_sig[e] = sgv[i];
                    if (k > best) { best = k; bidx = e; }
                }
            }
        }
        for (int r = 0; r < K; r++) {
            const unsigned mx = __reduce_max_sync(kFull, best);
            const unsigned win = __reduce_min_sync(kFull, best == mx ? (unsigned)bidx : 0xffffffffu);
            if (lane == 0) s_sel[r] = (int)win;
            if (lane == (int)(win & 31u)) {          // the winner's lane removes it and rescans
                s_key[win] = 0u;
                best = 0u;
                bidx = 0x7fffffff;
                for (int e = lane; e < E; e += 32) {
                    const unsigned k = s_key[e];
                    if (k > best) { best = k; bidx = e; }
                }
            }
        }
        __syncwarp();
        const int me = lane < K ? s_sel[lane] : 0;   // written by lane 0 of this warp
        const float sg = lane < K ? s_sig[me] : 0.0f;
        float sum = sg;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
        float den = sum + 1e-20f;
        if constexpr (V != 0) {
            if (d.score_func == MOE_SCORE_SOFTMAX) den = sum;   // the softmax family: no epsilon
        }
        const float mw = d.norm_topk ? d.scale * sg / den : d.scale * sg;
        if (lane < K) {
            s_slab[lane] = s_pslab[me];
            s_scale[lane] = s_pscale[me];
            s_w[lane] = mw;
        } else if (lane == K && d.n_shared) {
            s_slab[lane] = p.sh_slab;
            s_scale[lane] = p.sh_scale;
            s_w[lane] = 1.0f;
        }
        __syncwarp();
        if (lane == 0) {          // release the slot tables to the block
            __threadfence_block();
            s_flags[2] = 1;
        }
        mark(2);
        if (blockIdx.x == 0) {
            if (want_counts) {
                for (int e = lane; e < E; e += 32) p.ws.cnt[e] = 0;
                __syncwarp();
            }
            if (lane < K) {
                p.ws.topk_idx[lane] = me;
                p.ws.topk_w[lane] = mw;
                if (want_counts) p.ws.cnt[me] = 1;
            }
        }
    }
    // warps 1..7: wait (bounded) for the slot tables before the first routed unit
    bool routed = warp == 0;
    auto wait_routing = [&]() -> bool {
        if (routed) return true;
        int v = 1;
        if (lane == 0) {
            const unsigned long long t0 = now_ns();
            while ((v = s_flags[2]) == 0) {
                __nanosleep(64);
                if (now_ns() - t0 > kWaitNs) break;
            }
            if (v == 0) atomicOr(p.ws.err, kErrGrid);
        }
        v = __shfl_sync(kFull, v, 0);
        __threadfence_block();
        routed = v == 1;
        return routed;
    };

    // ---- phase 1: gate/up + SwiGLU ------------------------------------------------------
    mark(2);
    int corr[kPlanes] = {};
#pragma unroll
    for (int k = 0; k < CPLH; k++) {
        if (fullH || lane + 32 * k < C) {
            const int4 t = xdsum[lane + 32 * k];
            const int tv[3] = {t.x, t.y, t.z};
#pragma unroll
            for (int q = 0; q < kPlanes; q++) corr[q] -= 8 * tv[q];
        }
    }
    const uint32_t xdig_a = smem_u32(xdig) + (uint32_t)(lane * 16);
    auto gu_compute = [&](Unit u, const uint4 (&w2)[2 * CPLH], float sg, float su) {
        const int slot = u.pos < 0 ? K : u.pos, o = u.o;
        int lo[2][kPlanes], hi[2][kPlanes];
#pragma unroll
        for (int rr = 0; rr < 2; rr++)
#pragma unroll
            for (int q = 0; q < kPlanes; q++) { lo[rr][q] = corr[q]; hi[rr][q] = 0; }
#pragma unroll
        for (int k = 0; k < CPLH; k++) {
            if (fullH || lane + 32 * k < C) {
                uint4 dig[kQ];
#pragma unroll
                for (int q = 0; q < kQ; q++) dig[q] = lds128(xdig_a + (uint32_t)(q * C * 16 + 512 * k));
                const uint4 w[2] = {w2[k], w2[CPLH + k]};
                dot_rows<2>(w, dig, lo, hi);
            }
        }
        float v[2] = {planes_lh_to_float(lo[0], hi[0]), planes_lh_to_float(lo[1], hi[1])};
        const float tot = reduce_scatter<2>(v, lane);            // lane < 16: gate, else up
        const float up = __shfl_down_sync(kFull, tot, 16);
        if (lane == 0) p.ws.h[(size_t)slot * d.I_max + o] = silu_mul(tot * s_x * sg, up * s_x * su);
    };
    // the next unit's loads are in flight while this one is computed; the loop is kept
    // rolled (its body is large: unrolling it only grows the instruction footprint)
    if constexpr (V == 2) {
        int lo2[2][kPlanes], hi2[2][kPlanes];    // a unit's sums, carried between its segments
        auto step_compute = [&](Step st, const uint4 (&w2)[NBUF], float sg, float su, const uint32_t (&pr)[2 * CPLH]) {
            const bool i8 = is8(st.u);
            if (isg(st.u)) {
                float f[2] = {0.0f, 0.0f};
#pragma unroll
                for (int k = 0; k < CPLH; k++) {
                    if (fullH || lane + 32 * k < C) {
                        uint4 dig[kQ];
#pragma unroll
                        for (int q = 0; q < kQ; q++) dig[q] = lds128(xdig_a + (uint32_t)(q * C * 16 + 512 * k));
                        int lo[2][kPlanes] = {}, hi[2][kPlanes] = {};
                        const uint4 w[2] = {w2[k], w2[NBUF / 2 + k]};
                        dot_rows<2>(w, dig, lo, hi);
                        const int4 t = xdsum[lane + 32 * k];
                        const float xs = fmaf((float)t.y, 256.0f, (float)t.x);     // sum of the chunk's X
#pragma unroll
                        for (int rr = 0; rr < 2; rr++) {
                            const uint32_t pw = pr[rr * CPLH + k];
                            f[rr] = fmaf(g64_s(pw), planes_lh_to_float(lo[rr], hi[rr]), fmaf(g64_b(pw), xs, f[rr]));
                        }
                    }
                }
                const float tot = reduce_scatter<2>(f, lane);
                const float up = __shfl_down_sync(kFull, tot, 16);
                const int slot = st.u.pos < 0 ? K : st.u.pos;
                if (lane == 0) p.ws.h[(size_t)slot * d.I_max + st.u.o] = silu_mul(tot * s_x, up * s_x);
                return;
            }
            if (st.seg == 0) {
#pragma unroll
                for (int rr = 0; rr < 2; rr++)
#pragma unroll
                    for (int q = 0; q < kPlanes; q++) { lo2[rr][q] = i8 ? 0 : corr[q]; hi2[rr][q] = 0; }
            }
            if (!i8) {
#pragma unroll
                for (int k = 0; k < CPLH; k++) {
                    if (fullH || lane + 32 * k < C) {
                        uint4 dig[kQ];
#pragma unroll
                        for (int q = 0; q < kQ; q++) dig[q] = lds128(xdig_a + (uint32_t)(q * C * 16 + 512 * k));
                        const uint4 w[2] = {w2[k], w2[NBUF / 2 + k]};
                        dot_rows<2>(w, dig, lo2, hi2);
                    }
                }
            } else {
#pragma unroll
                for (int t = 0; t < SEG; t++) {
                    const int k = st.seg * SEG + t;
                    if (k < CPLH && (fullH || lane + 32 * k < C)) {
                        uint4 dig[kQ];
#pragma unroll
                        for (int q = 0; q < kQ; q++) dig[q] = lds128(xdig_a + (uint32_t)(q * C * 16 + 512 * k));
                        const uint4 w[2][2] = {{w2[2 * t], w2[2 * t + 1]}, {w2[NBUF / 2 + 2 * t], w2[NBUF / 2 + 2 * t + 1]}};
                        dot8_rows<2>(w, dig, lo2);
                    }
                }
            }
            if (i8 && st.seg == 0) return;       // the unit's second segment follows
            const int slot = st.u.pos < 0 ? K : st.u.pos;
            float v[2] = {planes_lh_to_float(lo2[0], hi2[0]), planes_lh_to_float(lo2[1], hi2[1])};
            const float tot = reduce_scatter<2>(v, lane);
            const float up = __shfl_down_sync(kFull, tot, 16);
            if (lane == 0) p.ws.h[(size_t)slot * d.I_max + st.u.o] = silu_mul(tot * s_x * sg, up * s_x * su);
        };
        if (!loaded && u_first.pos < K) {
            if (!wait_routing()) return;
            load_step(Step{u_first, 0}, wa, sga, sua, pra);
        }
#pragma unroll 1
        for (Step st = {u_first, 0}, sn; st.u.pos < K; st = sn) {
            sn = next_step(st);
            if (sn.u.pos < K) {
                if (sn.u.pos >= 0 && !wait_routing()) return;
                load_step(sn, wb, sgb, sub, prb);
            }
            step_compute(st, wa, sga, sua, pra);
#pragma unroll
            for (int k = 0; k < NBUF; k++) wa[k] = wb[k];
#pragma unroll
            for (int k = 0; k < 2 * CPLH; k++) pra[k] = prb[k];
            sga = sgb;
            sua = sub;
        }
    } else {
    if (!loaded && u_first.pos < K) {
        if (!wait_routing()) return;
        load_gu(u_first, wa, sga, sua);
    }
#pragma unroll 1
    for (Unit u = u_first, un; u.pos < K; u = un) {
        un = next_unit(u);
        if (un.pos < K) {
            if (un.pos >= 0 && !wait_routing()) return;
            load_gu(un, wb, sgb, sub);
        }
        gu_compute(u, wa, sga, sua);
#pragma unroll
        for (int k = 0; k < 2 * CPLH; k++) wa[k] = wb[k];
        sga = sgb;
        sua = sub;
        if (trace && warp == 0 && lane == 0) {    // warp 0 has routed units only
            const int i = (u.pos * d.I + u.o - gw) / nw;
            if (i < 32) tr[8 + i] = now_ns();
        }
    }
    }

    // ---- down: half-block hb (warps 4 hb .. 4 hb + 3) serves slot j; warp wl of the slot's
    // nwj warps takes row blocks wl, wl + nwj, ...  The first unit's loads go out before
    // barrier 2 (weights do not depend on h).
    if (!wait_routing()) return;     // the slot tables (on failure every warp returns here)
    const int hb = warp >> 2;
    const int hbg = 2 * blockIdx.x + hb;
    const int j = hbg % J;
    const int wl = (hbg / J) * 4 + (warp & 3);
    const int nwj = 4 * ((2 * G - 1 - j) / J + 1);
    // V == 2: an int8 slot's down rows (I bytes) are streamed one chunk (2 uint4 per row) per step
    constexpr int NBD = V == 2 ? (kDnRows * CPLI > 2 * kDnRows ? kDnRows * CPLI : 2 * kDnRows) : kDnRows * CPLI;
    const bool j8 = j == K ? s8 : r8;
    const bool jg = j == K ? sgf : rg;        // group-64 down rows: int4 layout, (s, b) per 64 inputs
    const uint8_t *dslab = s_slab[j] + (size_t)(j8 ? 2 : 1) * d.I * d.H;
    const float *sd = s_scale[j] + 2 * d.I;
    const bool dn_writer = (lane & 7) == 0;                // lane l ends with row l / 8
    auto load_dn8 = [&](int rb, int kc, uint4 (&w)[NBD], float &sc) {
        const int c = lane + 32 * kc;
        if (fullI || c < Cd) {
#pragma unroll
            for (int rr = 0; rr < kDnRows; rr++) {
                const uint4 *row = reinterpret_cast<const uint4 *>(dslab + (size_t)(rb * kDnRows + rr) * d.I);
                w[2 * rr] = ldg_stream(row + 2 * c);
                w[2 * rr + 1] = ldg_stream(row + 2 * c + 1);
            }
        }
        if (dn_writer) sc = __ldg(sd + rb * kDnRows + (lane >> 3));
    };
    auto load_dn = [&](int rb, uint4 (&w)[NBD], float &sc) {
        const uint4 *src = reinterpret_cast<const uint4 *>(dslab + (size_t)rb * kDnRows * sh.drowbytes) + lane;
#pragma unroll
        for (int rr = 0; rr < kDnRows; rr++)
#pragma unroll
            for (int k = 0; k < CPLI; k++)
                if (fullI || lane + 32 * k < Cd) w[rr * CPLI + k] = ldg_stream(src + rr * (sh.drowbytes / 16) + 32 * k);
        if (dn_writer) sc = __ldg(sd + rb * kDnRows + (lane >> 3));
    };
    auto load_dpairs = [&](int rb, uint32_t (&pd)[kDnRows * CPLI]) {
        const uint32_t *pw = reinterpret_cast<const uint32_t *>(s_scale[j]) + (size_t)2 * d.I * (H / 64);
        const int ng = d.I / 64;
#pragma unroll
        for (int rr = 0; rr < kDnRows; rr++)
#pragma unroll
            for (int k = 0; k < CPLI; k++) {
                const int c = lane + 32 * k;
                if (fullI || c < Cd) pd[rr * CPLI + k] = __ldg(pw + (size_t)(rb * kDnRows + rr) * ng + (c >> 1));
            }
    };
    uint32_t pda[kDnRows * CPLI], pdb[kDnRows * CPLI];   // V == 2, group-64 slot: pairs of the buffered unit
    uint4 da[NBD], db[NBD];
    float sca = 0.0f, scb = 0.0f;
    if (wl < sh.RB) {
        if (V == 2 && j8) load_dn8(wl, 0, da, sca);
        else load_dn(wl, da, sca);
        if (V == 2 && jg) load_dpairs(wl, pda);
    }

    // ---- barrier 2: every SwiGLU activation is written ------------------------------------
    if (!grid_barrier(bar2, target, p.ws.err, s_flags + 1)) return;
    if (blockIdx.x == 0 && tid == 0) *reinterpret_cast<volatile unsigned *>(epoch) = gen;
    mark(3);

    // ---- phase 2: the half-block loads slot j's h (thread t of the half: chunk t), takes
    // max |h|, and writes the digits to shared memory (x digits are no longer read)
    const int ht = tid & 127;
    const bool hchunk = ht < Cd;
    float hv[32];
    {
        const float4 *h4 = reinterpret_cast<const float4 *>(p.ws.h + (size_t)j * d.I_max + (size_t)(hchunk ? ht : 0) * 32);
#pragma unroll
        for (int t = 0; t < 8; t++) {
            const float4 f = hchunk ? __ldcg(h4 + t) : make_float4(0.f, 0.f, 0.f, 0.f);
            hv[4 * t] = f.x; hv[4 * t + 1] = f.y; hv[4 * t + 2] = f.z; hv[4 * t + 3] = f.w;
        }
    }
    float hm = 0.0f;
    bool hnan = false;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        hm = fmaxf(hm, fabsf(hv[i]));
        hnan |= isnan(hv[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hm = fmaxf(hm, __shfl_xor_sync(kFull, hm, o));
    hnan = __any_sync(kFull, hnan);
    if (lane == 0) red[56 + warp] = hnan ? __int_as_float(0x7fc00000) : hm;
    named_barrier(1 + hb, 128);
    float hmax = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; w++) {
        const float r4 = red[56 + 4 * hb + w];
        hmax = (isnan(r4) || isnan(hmax)) ? r4 + hmax : fmaxf(hmax, r4);
    }
    const float hs = hmax / kQMax;                    // NaN propagates
    const float hinv = (hs > 0.0f && isfinite(hs)) ? 1.0f / hs : 0.0f;
    const float coef_j = s_w[j] * hs;
    uint4 *hd = xdig + (size_t)hb * (kQ + 1) * Cd;
    if (hchunk) {
        uint4 dig[kQ];
        int ds[kPlanes];
        quant_chunk(hv, hinv, dig, ds);
#pragma unroll
        for (int q = 0; q < kQ; q++) hd[q * Cd + ht] = dig[q];
        hd[kQ * Cd + ht] = make_uint4((unsigned)ds[0], (unsigned)ds[1], kPlanes > 2 ? (unsigned)ds[kPlanes - 1] : 0u, 0u);
    }
    named_barrier(1 + hb, 128);
    mark(4);
    uint4 hdig[CPLI][kQ];
    int dcorr[kPlanes] = {};
#pragma unroll
    for (int k = 0; k < CPLI; k++) {
        const int c = lane + 32 * k;
        if (fullI || c < Cd) {
#pragma unroll
            for (int q = 0; q < kQ; q++) hdig[k][q] = hd[q * Cd + c];
            const uint4 t = hd[kQ * Cd + c];
            const int tv[3] = {(int)t.x, (int)t.y, (int)t.z};
#pragma unroll
            for (int q = 0; q < kPlanes; q++) dcorr[q] -= 8 * tv[q];
        } else {
#pragma unroll
            for (int q = 0; q < kQ; q++) hdig[k][q] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    auto dn_compute = [&](int rb, const uint4 (&w2)[NBD], float sc) {
        int lo[kDnRows][kPlanes], hi[kDnRows][kPlanes];
#pragma unroll
        for (int rr = 0; rr < kDnRows; rr++)
#pragma unroll
            for (int q = 0; q < kPlanes; q++) { lo[rr][q] = dcorr[q]; hi[rr][q] = 0; }
#pragma unroll
        for (int k = 0; k < CPLI; k++) {
            if (fullI || lane + 32 * k < Cd) {
                uint4 w[kDnRows];
#pragma unroll
                for (int rr = 0; rr < kDnRows; rr++) w[rr] = w2[rr * CPLI + k];
                dot_rows<kDnRows>(w, hdig[k], lo, hi);
            }
        }
        float v[kDnRows];
#pragma unroll
        for (int rr = 0; rr < kDnRows; rr++) v[rr] = planes_lh_to_float(lo[rr], hi[rr]);
        const float tot = reduce_scatter<kDnRows>(v, lane);
        if (dn_writer) p.ws.dpart[(size_t)j * H + rb * kDnRows + (lane >> 3)] = tot * coef_j * sc;
    };
    if (V == 2 && j8) {
        // int8 down rows: steps (rb, chunk kc), the sums of a row block carried over its chunks
        int lo8[kDnRows][kPlanes], hi8[kDnRows][kPlanes];
#pragma unroll 1
        for (int rb = wl, kc = 0; rb < sh.RB;) {
            const int kn = kc + 1 < CPLI ? kc + 1 : 0, rn = kc + 1 < CPLI ? rb : rb + nwj;
            if (rn < sh.RB) load_dn8(rn, kn, db, scb);
            if (kc == 0) {
#pragma unroll
                for (int rr = 0; rr < kDnRows; rr++)
#pragma unroll
                    for (int q = 0; q < kPlanes; q++) { lo8[rr][q] = 0; hi8[rr][q] = 0; }
            }
#pragma unroll
            for (int k = 0; k < CPLI; k++) {
                if (k == kc && (fullI || lane + 32 * k < Cd)) {
                    const uint4 w[kDnRows][2] = {{da[0], da[1]}, {da[2], da[3]}, {da[4], da[5]}, {da[6], da[7]}};
                    dot8_rows<kDnRows>(w, hdig[k], lo8);
                }
            }
            if (kc + 1 == CPLI) {
                float v[kDnRows];
#pragma unroll
                for (int rr = 0; rr < kDnRows; rr++) v[rr] = planes_lh_to_float(lo8[rr], hi8[rr]);
                const float tot = reduce_scatter<kDnRows>(v, lane);
                if (dn_writer) p.ws.dpart[(size_t)j * H + rb * kDnRows + (lane >> 3)] = tot * coef_j * sca;
            }
#pragma unroll
            for (int k = 0; k < NBD; k++) da[k] = db[k];
            sca = scb;
            rb = rn;
            kc = kn;
        }
    } else if (V == 2 && jg) {
        // group-64 down rows: per chunk, s sum(u X) + b sum(X) with the chunk's h digit sums
        float xsh[CPLI];
#pragma unroll
        for (int k = 0; k < CPLI; k++) {
            const int c = lane + 32 * k;
            const uint4 t = (fullI || c < Cd) ? hd[kQ * Cd + c] : make_uint4(0u, 0u, 0u, 0u);
            xsh[k] = fmaf((float)(int)t.y, 256.0f, (float)(int)t.x);
        }
#pragma unroll 1
        for (int rb = wl; rb < sh.RB; rb += nwj) {
            const int rn = rb + nwj;
            if (rn < sh.RB) {
                load_dn(rn, db, scb);
                load_dpairs(rn, pdb);
            }
            float f[kDnRows] = {};
#pragma unroll
            for (int k = 0; k < CPLI; k++) {
                if (fullI || lane + 32 * k < Cd) {
                    int lo[kDnRows][kPlanes] = {}, hi[kDnRows][kPlanes] = {};
                    uint4 w[kDnRows];
#pragma unroll
                    for (int rr = 0; rr < kDnRows; rr++) w[rr] = da[rr * CPLI + k];
                    dot_rows<kDnRows>(w, hdig[k], lo, hi);
#pragma unroll
                    for (int rr = 0; rr < kDnRows; rr++) {
                        const uint32_t pw = pda[rr * CPLI + k];
                        f[rr] = fmaf(g64_s(pw), planes_lh_to_float(lo[rr], hi[rr]), fmaf(g64_b(pw), xsh[k], f[rr]));
                    }
                }
            }
            const float tot = reduce_scatter<kDnRows>(f, lane);
            if (dn_writer) p.ws.dpart[(size_t)j * H + rb * kDnRows + (lane >> 3)] = tot * coef_j;
#pragma unroll
            for (int k = 0; k < NBD; k++) da[k] = db[k];
#pragma unroll
            for (int k = 0; k < kDnRows * CPLI; k++) pda[k] = pdb[k];
        }
    } else
#pragma unroll 1
    for (int rb = wl; rb < sh.RB; rb += nwj) {
        const int rn = rb + nwj;
        if (rn < sh.RB) load_dn(rn, db, scb);             // in flight during this unit
        dn_compute(rb, da, sca);
#pragma unroll
        for (int k = 0; k < NBD; k++) da[k] = db[k];
        sca = scb;
        if (trace && warp == 0 && lane == 0) {
            const int i = (rb - wl) / nwj;
            if (i < 24) tr[40 + i] = now_ns();
        }
    }

    // ---- barrier 3, then phase 3: combine ---------------------------------------------------
    if (!grid_barrier(bar3, target, p.ws.err, s_flags + 1)) return;
    mark(5);
    for (int o = blockIdx.x * kThreads + tid; o < H; o += G * kThreads) {
        float acc = 0.0f;
        for (int k = 0; k < K; k++) acc += __ldcg(p.ws.dpart + (size_t)k * H + o);
        if (d.n_shared) acc += __ldcg(p.ws.dpart + (size_t)K * H + o);
        y[o] = d.prenorm ? x[o] + acc : acc;
    }
    mark(6);
}

constexpr int kMaxCplH = 8;   // H up to 8192
constexpr int kMaxCplI = 2;   // I up to 2048 (digits of more chunks do not fit in registers)

template <int A, int B, int V>
cudaError_t launch_t(cudaLaunchConfig_t &cfg, const Params &p, const float *x, float *y, const FusedShape &s,
                     int counts) {
    return cudaLaunchKernelEx(&cfg, decode_fused_kernel<A, B, V>, p, x, y, s, counts);
}

template <int B, int V>
cudaError_t launch_h(int a, cudaLaunchConfig_t &cfg, const Params &p, const float *x, float *y,
                     const FusedShape &s, int counts) {
    switch (a) {
        case 1: return launch_t<1, B, V>(cfg, p, x, y, s, counts);
        case 2: return launch_t<2, B, V>(cfg, p, x, y, s, counts);
        case 3: return launch_t<3, B, V>(cfg, p, x, y, s, counts);
        case 4: return launch_t<4, B, V>(cfg, p, x, y, s, counts);
        case 6: return launch_t<6, B, V>(cfg, p, x, y, s, counts);
        case 8: return launch_t<8, B, V>(cfg, p, x, y, s, counts);
    }
    return cudaErrorInvalidValue;
}

// the instantiation a handle needs: 2 with an int8 expert, 1 for the routing variants
// (group-limited or softmax selection), else 0
int kernel_variant(const Dims &d) {
    if (d.mma_fmt) return 2;
    return (d.n_group > 1 || d.score_func == MOE_SCORE_SOFTMAX) ? 1 : 0;
}

int cpl_h(const Dims &d) {
    const int c = (d.H / 32 + 31) / 32;
    return c == 5 ? 6 : (c == 7 ? 8 : c);       // instantiated: 1, 2, 3, 4, 6, 8
}

template <int A, int B, int V>
cudaError_t attr_t() {
    cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<A, B, V>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget);
    int nb = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, decode_fused_kernel<A, B, V>, kThreads, kSmemBudget);
    if (e == cudaSuccess && nb < 1) e = cudaErrorInvalidConfiguration;
    return e;
}

}  // namespace

int decode_grid_blocks(const Dims &d) { return d.dec_grid; }

bool decode_fast_supported(const Dims &d) {                                             // int8 experts: tensor-core kernels
    if (d.H % kDnRows != 0 || d.H % 32 != 0 || d.I % 32 != 0) return false;
    if (d.n_shared && d.I_sh != d.I) return false;
    if (d.K + d.n_shared > kMaxSlots || d.K + d.n_shared > 32 || d.E > 1024) return false;
    if ((d.H / 32 + 31) / 32 > kMaxCplH || (d.I / 32 + 31) / 32 > kMaxCplI) return false;
    return fused_shape(d).smem <= (size_t)kSmemBudget;
}

// Kernel attributes and this GPU's grid (one block per SM) for a handle; a GPU
// with too few SMs for the slots runs the generic kernels instead (d.fast_decode
// cleared).
cudaError_t prepare_decode_fast(Dims &d) {
    d.dec_grid = 0;
    if (!d.fast_decode) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // every slot needs at least one half-block in the down phase
    if (2 * sms < d.K + d.n_shared) {
        d.fast_decode = 0;
        return cudaSuccess;
    }
    // every instantiation gets the same (largest) shared-memory limit, so
    // handles of different shapes coexist
    const int b = (d.I / 32 + 31) / 32;
    switch (cpl_h(d) * 16 + b * 4 + kernel_variant(d)) {
#define MOE_ATTR(A, B) case A * 16 + B * 4: e = attr_t<A, B, 0>(); break; \
                       case A * 16 + B * 4 + 1: e = attr_t<A, B, 1>(); break; \
                       case A * 16 + B * 4 + 2: e = attr_t<A, B, 2>(); break;
        MOE_ATTR(1, 1) MOE_ATTR(2, 1) MOE_ATTR(3, 1) MOE_ATTR(4, 1) MOE_ATTR(6, 1) MOE_ATTR(8, 1)
        MOE_ATTR(1, 2) MOE_ATTR(2, 2) MOE_ATTR(3, 2) MOE_ATTR(4, 2) MOE_ATTR(6, 2) MOE_ATTR(8, 2)
#undef MOE_ATTR
        default: e = cudaErrorInvalidValue;
    }
    if (e == cudaSuccess) d.dec_grid = sms;
    return e;
}

// One launch for the whole T == 1 step.  ev (optional): ev[0],
// ev[1] before the kernel, ev[2..4] after it (stage 1 = the fused kernel).
cudaError_t launch_decode_fast(const Params &p, const float *x, float *y, cudaStream_t st, cudaEvent_t *ev,
                               bool want_counts) {
    const FusedShape s = fused_shape(p.d);
    // programmatic stream serialisation: the kernel may be launched before the previous kernel
    // on the stream ends (its blocks take each SM as the previous kernel's block there exits),
    // and waits for that kernel (griddepcontrol.wait) before it reads x or the workspace.  The
    // grid is one block per SM and the blocks meet at grid barriers, so all of them must be
    // resident together: true on a GPU this call has to itself (one block fills an SM's
    // registers); a cooperative launch would guarantee it but is never started early (measured
    // on the GLM-5.2 layer, calls back to back: 44.0 us per call cooperative, 40.7 us with the
    // early launch).  When other work holds SMs, a block that cannot start makes the barrier
    // waits run out (bounded), and the call reports it through moe_device_error.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    if (p.d.dec_grid < 1) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(p.d.dec_grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = s.smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaSuccess;
    if (ev) e = cudaEventRecord(ev[0], st);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[1], st);
    if (e != cudaSuccess) return e;
    const int b = (p.d.I / 32 + 31) / 32;
    const int counts = want_counts ? 1 : 0;
    const int a = cpl_h(p.d);
    switch (kernel_variant(p.d)) {
        case 0: e = b == 1 ? launch_h<1, 0>(a, cfg, p, x, y, s, counts) : launch_h<2, 0>(a, cfg, p, x, y, s, counts); break;
        case 1: e = b == 1 ? launch_h<1, 1>(a, cfg, p, x, y, s, counts) : launch_h<2, 1>(a, cfg, p, x, y, s, counts); break;
        default: e = b == 1 ? launch_h<1, 2>(a, cfg, p, x, y, s, counts) : launch_h<2, 2>(a, cfg, p, x, y, s, counts);
    }
    for (int i = 2; ev && e == cudaSuccess && i < 5; i++) e = cudaEventRecord(ev[i], st);
    return e;
}

}  // namespace moe
