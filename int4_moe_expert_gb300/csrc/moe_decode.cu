// Decode (T == 1) streaming path: gate/up + SwiGLU and down as persistent
// kernels in which every warp streams its own units of expert rows into
// shared memory with cp.async (two buffers per warp: one is computed while
// the next one lands), followed by a small combine kernel.  The three are
// chained with programmatic dependent launch after the router.
//
// What is computed is the same as the generic kernels (reader.mx
// "25GB 内存上运行 GLM 5.2 744B" section 11; devpress GLM-5.2 breakdown
// "Step 6 (MoE)" 6b-6d):  g = s_g (Q_g x), u = s_u (Q_u x), h = silu(g) u,
// d = s_d (Q_d h), y = sum_k w_k d_k + d_shared.
//
// Arithmetic.  An activation vector v (x, or one expert's h) is held as
// 24-bit fixed point with one scale per vector: X_i = rint(v_i / s),
// s = max|v| / 8355711, |X_i| <= 8355711 = 0x7F7F7F, written as three signed
// base-256 digits X = d2 65536 + d1 256 + d0, each in [-128, 127].  A packed
// int4 weight byte holds two unsigned nibbles n = q + 8 (section 06 format),
// so one row's dot product is
//     sum_i q_i v_i = s * sum_p 256^p (sum_i n_i d_{p,i} - 8 sum_i d_{p,i}),
// with every inner sum exact in int32 (dp4a: four unsigned nibble bytes times
// four signed digit bytes).  Only the final plane combination and the scale
// are floating point.  The representation error of v is at most
// max|v| * 2^-24 per element, the same order as one float32 rounding.
//
// Layout of a vector's digits (shared memory): for chunk c (elements
// 32c..32c+31, one 16-byte weight load) and q = 2p + lh, the uint4 at
// [q * C + c] holds, in word m, the plane-p digits of elements 8m+{0,2,4,6}
// (lh = 0: the low nibbles of word m) or 8m+{1,3,5,7} (lh = 1: the high
// nibbles), one per byte, matching the nibble order of the weight word.
//
// Why cp.async and not bulk (TMA) copies: measured on this GPU, one block
// issuing 1-D bulk copies completes about one copy per 0.27 us whatever its
// size, so 6-12 KB units capped a block at 23-45 GB/s; per-lane 16-byte
// asynchronous copies from eight warps keep enough bytes in flight.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kGuRows = 2;          // row pairs (gate + up) per gate/up unit
constexpr int kDnRows = 8;          // output rows per down unit
constexpr int kBufs = 2;            // gate/up buffers per warp
constexpr int kGuSmemBudget = 220 * 1024;
constexpr int kDnSmemBudget = 220 * 1024;
constexpr float kQMax = 8355711.0f;         // 0x7F7F7F

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void dp4a_us(int &acc, uint32_t nib, uint32_t dig) {
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(nib), "r"(dig));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int m) {
    return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// acc[p] += sum over the 32 weights of one 16-byte chunk of nibble * digit(p)
__device__ __forceinline__ void dot_chunk(const uint4 w, const uint4 (&dig)[6], int (&acc)[3]) {
#pragma unroll
    for (int m = 0; m < 4; m++) {
        const uint32_t word = word_of(w, m);
        const uint32_t lo = word & 0x0F0F0F0Fu;
        const uint32_t hi = (word >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int p = 0; p < 3; p++) {
            dp4a_us(acc[p], lo, word_of(dig[2 * p], m));
            dp4a_us(acc[p], hi, word_of(dig[2 * p + 1], m));
        }
    }
}

// Same sums with the high nibbles kept in place (byte value 16 n): acc_lo
// collects n * d for the low nibbles, acc_hi 16 n * d for the high ones, so
// the total is acc_lo + acc_hi / 16 (exact: acc_hi is a multiple of 16).
__device__ __forceinline__ void dot_chunk_lh(const uint4 w, const uint4 (&dig)[6], int (&lo_acc)[3],
                                             int (&hi_acc)[3]) {
#pragma unroll
    for (int m = 0; m < 4; m++) {
        const uint32_t word = word_of(w, m);
        const uint32_t lo = word & 0x0F0F0F0Fu;
        const uint32_t hi = word & 0xF0F0F0F0u;
#pragma unroll
        for (int p = 0; p < 3; p++) {
            dp4a_us(lo_acc[p], lo, word_of(dig[2 * p], m));
            dp4a_us(hi_acc[p], hi, word_of(dig[2 * p + 1], m));
        }
    }
}

__device__ __forceinline__ float planes_lh_to_float(const int (&lo)[3], const int (&hi)[3]) {
    const int a0 = lo[0] + (hi[0] >> 4), a1 = lo[1] + (hi[1] >> 4), a2 = lo[2] + (hi[2] >> 4);
    return fmaf(__int2float_rn(a2), 65536.0f, fmaf(__int2float_rn(a1), 256.0f, __int2float_rn(a0)));
}

__device__ __forceinline__ float planes_to_float(const int (&a)[3]) {
    return fmaf(__int2float_rn(a[2]), 65536.0f, fmaf(__int2float_rn(a[1]), 256.0f, __int2float_rn(a[0])));
}

// Digits of the 32 values of one chunk (natural order) scaled by inv = 1/s;
// dsum[p] = sum of the plane-p digits.
__device__ __forceinline__ void quant_chunk(const float (&v)[32], float inv, uint4 (&dig)[6], int (&dsum)[3]) {
    uint32_t w[6][4];
#pragma unroll
    for (int q = 0; q < 6; q++)
#pragma unroll
        for (int m = 0; m < 4; m++) w[q][m] = 0u;
    dsum[0] = dsum[1] = dsum[2] = 0;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        int X = __float2int_rn(v[i] * inv);
        X = min(max(X, -8355711), 8355711);
        const int d0 = ((X + 128) & 255) - 128;
        const int X1 = (X - d0) >> 8;
        const int d1 = ((X1 + 128) & 255) - 128;
        const int d2 = (X1 - d1) >> 8;
        const int m = i >> 3, e = i & 7, lh = e & 1, b = e >> 1;
        w[0 + lh][m] |= (uint32_t)(d0 & 255) << (8 * b);
        w[2 + lh][m] |= (uint32_t)(d1 & 255) << (8 * b);
        w[4 + lh][m] |= (uint32_t)(d2 & 255) << (8 * b);
        dsum[0] += d0;
        dsum[1] += d1;
        dsum[2] += d2;
    }
#pragma unroll
    for (int q = 0; q < 6; q++) dig[q] = make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
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

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }


// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------

struct GuShape {
    int C;            // chunks per row = H / 32
    int rowbytes;     // H / 2
    int unit_bytes;   // 2 * kGuRows * rowbytes
    int U_sh, U_r;    // units of the shared expert, units per routed expert
    int units;
    size_t smem;
};

// smem: [kWarps][kBufs][unit_bytes] | xdig [6][C] uint4 | xdsum [C] int4 | red
__host__ __device__ inline GuShape gu_shape(const Dims &d) {
    GuShape s;
    s.C = d.H / 32;
    s.rowbytes = d.H / 2;
    s.unit_bytes = 2 * kGuRows * s.rowbytes;
    s.U_sh = d.n_shared ? d.I_sh / kGuRows : 0;
    s.U_r = d.I / kGuRows;
    s.units = s.U_sh + d.K * s.U_r;
    s.smem = (size_t)kWarps * kBufs * s.unit_bytes + (size_t)7 * s.C * 16 + 64 * sizeof(float);
    return s;
}

// Pointers of slot j (j < K: the j-th routed choice; j == K: shared expert)
// for lane j of the calling warp; read after the routing is final.
struct SlotPtr {
    const uint8_t *slab;
    const float *scale;
};
__device__ __forceinline__ SlotPtr lane_slot(const Params &p, int lane) {
    SlotPtr r{nullptr, nullptr};
    if (lane < p.d.K) {
        const int e = __ldcg(p.ws.topk_idx + lane);
        r.slab = p.slabs[e];
        r.scale = p.scales[e];
    } else if (lane == p.d.K && p.d.n_shared) {
        r.slab = p.sh_slab;
        r.scale = p.sh_scale;
    }
    return r;
}
__device__ __forceinline__ const void *shfl_ptr(const void *ptr, int src) {
    const unsigned long long v = reinterpret_cast<unsigned long long>(ptr);
    return reinterpret_cast<const void *>(__shfl_sync(0xffffffffu, v, src));
}

// CPL = chunks per lane = ceil(C / 32); lane l owns chunks l + 32 k.
template <int CPL>
__global__ void __launch_bounds__(kThreads, 1) gateup_stream_kernel(Params p, const float *__restrict__ x,
                                                                    GuShape sh) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint4 *xdig = reinterpret_cast<uint4 *>(smem + (size_t)kWarps * kBufs * sh.unit_bytes);
    int4 *xdsum = reinterpret_cast<int4 *>(xdig + 6 * sh.C);
    float *red = reinterpret_cast<float *>(xdsum + sh.C);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Dims &d = p.d;
    const int H = d.H, C = sh.C;
    const bool full_lanes = (C % 32) == 0;
    const uint32_t wbuf = smem_u32(smem + (size_t)warp * kBufs * sh.unit_bytes) + (uint32_t)(lane * 16);

    // units of this warp: u = gw, gw + nw, ...; the shared expert's come first
    const int nw = gridDim.x * kWarps;
    const int gw = blockIdx.x * kWarps + warp;
    bool routed_ready = false;
    SlotPtr mine{nullptr, nullptr};

    auto unit_src = [&](int u, int &slot, int &rb, const uint8_t *&slab, const float *&scale, int &Ij) {
        if (u < sh.U_sh) {
            slot = d.K; rb = u; slab = p.sh_slab; scale = p.sh_scale; Ij = d.I_sh;
        } else {
            if (!routed_ready) {
                pdl_wait();
                mine = lane_slot(p, lane);
                routed_ready = true;
            }
            const int v = u - sh.U_sh;
            slot = v / sh.U_r;
            rb = v - slot * sh.U_r;
            slab = static_cast<const uint8_t *>(shfl_ptr(mine.slab, slot));
            scale = static_cast<const float *>(shfl_ptr(mine.scale, slot));
            Ij = d.I;
        }
    };
    // each lane copies the 16-byte pieces it will read itself
    auto issue = [&](int u, int buf) {
        int slot, rb, Ij;
        const uint8_t *slab;
        const float *scale;
        unit_src(u, slot, rb, slab, scale, Ij);
        const uint32_t dst = wbuf + (uint32_t)(buf * sh.unit_bytes);
        const uint8_t *gsrc = slab + (size_t)rb * kGuRows * sh.rowbytes + lane * 16;
        const uint8_t *usrc = slab + ((size_t)Ij + (size_t)rb * kGuRows) * sh.rowbytes + lane * 16;
#pragma unroll
        for (int rr = 0; rr < 2 * kGuRows; rr++) {
            const uint8_t *src = (rr < kGuRows ? gsrc + rr * sh.rowbytes : usrc + (rr - kGuRows) * sh.rowbytes);
            const uint32_t drow = dst + (uint32_t)(rr * sh.rowbytes);
#pragma unroll
            for (int k = 0; k < CPL; k++)
                if (full_lanes || lane + 32 * k < C) cp_async16(drow + 512 * k, src + 512 * k);
        }
    };

#pragma unroll
    for (int b = 0; b < kBufs; b++) {
        if (gw + b * nw < sh.units) issue(gw + b * nw, b);
        cp_async_commit();
    }

    // ---- quantise x once per block ----------------------------------------------
    float amax = 0.0f, ss = 0.0f;
    bool bad = false;
    for (int c = threadIdx.x; c < C; c += kThreads) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x + (size_t)c * 32);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const float4 v = __ldg(x4 + k);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
            bad |= !(isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        red[warp] = amax;
        red[kWarps + warp] = ss;
        red[2 * kWarps + warp] = bad ? 1.0f : 0.0f;
    }
    __syncthreads();
    amax = 0.0f;
    ss = 0.0f;
    bad = false;
    for (int w = 0; w < kWarps; w++) {
        amax = fmaxf(amax, red[w]);
        ss += red[kWarps + w];
        bad |= red[2 * kWarps + w] != 0.0f;
    }
    const float r = d.prenorm ? 1.0f / sqrtf(ss / (float)H + d.eps) : 1.0f;
    const float m = amax * r;
    const float s_x = bad ? __int_as_float(0x7fc00000) : m / kQMax;
    const float inv = (m > 0.0f && !bad) ? kQMax / m : 0.0f;
    for (int c = threadIdx.x; c < C; c += kThreads) {
        float v[32];
        const float4 *x4 = reinterpret_cast<const float4 *>(x + (size_t)c * 32);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const float4 f = __ldg(x4 + k);
            v[4 * k] = f.x * r; v[4 * k + 1] = f.y * r; v[4 * k + 2] = f.z * r; v[4 * k + 3] = f.w * r;
        }
        uint4 dig[6];
        int ds[3];
        quant_chunk(v, inv, dig, ds);
#pragma unroll
        for (int q = 0; q < 6; q++) xdig[q * C + c] = dig[q];
        xdsum[c] = make_int4(ds[0], ds[1], ds[2], 0);
    }
    __syncthreads();
    // per-lane correction: -8 * (sum of digits over this lane's chunks)
    int corr[3] = {0, 0, 0};
#pragma unroll
    for (int k = 0; k < CPL; k++) {
        if (full_lanes || lane + 32 * k < C) {
            const int4 t = xdsum[lane + 32 * k];
            corr[0] -= 8 * t.x; corr[1] -= 8 * t.y; corr[2] -= 8 * t.z;
        }
    }
    const uint32_t xdig_a = smem_u32(xdig) + (uint32_t)(lane * 16);

    // ---- stream units ---------------------------------------------------------------
    // lane l ends with row l / 8 of the unit: rows 0..kGuRows-1 gate, then up
    const bool writer = lane < 16 && (lane & 7) == 0;
    int buf = 0;
    for (int u = gw; u < sh.units; u += nw, buf = (buf + 1 == kBufs) ? 0 : buf + 1) {
        int slot, rb, Ij;
        const uint8_t *slab;
        const float *scale;
        unit_src(u, slot, rb, slab, scale, Ij);
        const int o = rb * kGuRows + (lane >> 3);
        float sg = 0.0f, su = 0.0f;
        if (writer) {            // issued now, needed after the dot products
            sg = __ldg(scale + o);
            su = __ldg(scale + Ij + o);
        }
        cp_async_wait_1();       // this unit's copies (this lane's own pieces) have landed
        const uint32_t st = wbuf + (uint32_t)(buf * sh.unit_bytes);
        int lo[2 * kGuRows][3], hi[2 * kGuRows][3];
        static_assert(kBufs == 2, "wait_group count below assumes two buffers");
#pragma unroll
        for (int rr = 0; rr < 2 * kGuRows; rr++) {
            lo[rr][0] = corr[0]; lo[rr][1] = corr[1]; lo[rr][2] = corr[2];
            hi[rr][0] = 0; hi[rr][1] = 0; hi[rr][2] = 0;
        }
#pragma unroll
        for (int k = 0; k < CPL; k++) {
            if (full_lanes || lane + 32 * k < C) {
                uint4 dig[6];
#pragma unroll
                for (int q = 0; q < 6; q++) dig[q] = lds128(xdig_a + (uint32_t)(q * C * 16 + 512 * k));
#pragma unroll
                for (int rr = 0; rr < 2 * kGuRows; rr++) {
                    const uint4 w = lds128(st + (uint32_t)(rr * sh.rowbytes + 512 * k));
                    dot_chunk_lh(w, dig, lo[rr], hi[rr]);
                }
            }
        }
        float v[2 * kGuRows];
#pragma unroll
        for (int rr = 0; rr < 2 * kGuRows; rr++) v[rr] = planes_lh_to_float(lo[rr], hi[rr]);
        const float tot = reduce_scatter<2 * kGuRows>(v, lane);
        const float up = __shfl_down_sync(0xffffffffu, tot, 16);   // up row of the same output
        if (writer) {
            const float hv = silu_mul(tot * s_x * sg, up * s_x * su);
            p.ws.h[(size_t)slot * d.I_max + o] = hv;
            atomicMax(p.ws.hmax + slot, __float_as_uint(fabsf(hv)));
        }
        // this buffer is free again: fetch the unit kBufs ahead into it
        if (u + kBufs * nw < sh.units) issue(u + kBufs * nw, buf);
        cp_async_commit();
    }
    cp_async_wait_0();
    if (!routed_ready) pdl_wait();
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// down: per-slot outputs times the routing weight, combined after.  Each warp
// works on one slot only, so its lanes keep that slot's h digits in registers.
// ---------------------------------------------------------------------------

constexpr int kDnBufs = 3;         // down buffers per warp

struct DnShape {
    int C;            // chunks per row = I / 32
    int rowbytes;     // I / 2
    int unit_bytes;   // kDnRows * rowbytes
    int J;            // slots (K + n_shared)
    int RB;           // row blocks = H / kDnRows
    size_t smem;
};

// smem: [kWarps][kDnBufs][unit_bytes]
__host__ __device__ inline DnShape dn_shape(const Dims &d) {
    DnShape s;
    s.C = d.I / 32;
    s.rowbytes = d.I / 2;
    s.unit_bytes = kDnRows * s.rowbytes;
    s.J = d.K + d.n_shared;
    s.RB = d.H / kDnRows;
    s.smem = (size_t)kWarps * kDnBufs * s.unit_bytes + 64;
    return s;
}

template <int CPL>
__global__ void __launch_bounds__(kThreads, 1) down_stream_kernel(Params p, DnShape sh) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Dims &d = p.d;
    const int H = d.H, K = d.K, J = sh.J, C = sh.C;
    const bool full_lanes = (C % 32) == 0;
    const uint32_t wbuf = smem_u32(smem + (size_t)warp * kDnBufs * sh.unit_bytes) + (uint32_t)(lane * 16);

    // warp gw serves slot j = gw % J; the warps of one slot split its row blocks
    const int nw = gridDim.x * kWarps;
    const int gw = blockIdx.x * kWarps + warp;
    const int j = gw % J;
    const int q = gw / J;
    const int nq = (nw - j + J - 1) / J;    // warps serving slot j

    pdl_trigger();   // the combine grid may launch; it waits for this one
    // Routing was final before the gate/up grid let this grid start, so the
    // weights can stream while the SwiGLU activations are still being made.
    const SlotPtr mine = lane_slot(p, lane);
    const uint8_t *dslab = static_cast<const uint8_t *>(shfl_ptr(mine.slab, j)) + (size_t)d.I * d.H + lane * 16;
    const float *sd = static_cast<const float *>(shfl_ptr(mine.scale, j)) + 2 * d.I;
    auto issue = [&](int rb, int buf) {
        const uint8_t *src = dslab + (size_t)rb * kDnRows * sh.rowbytes;
        const uint32_t dst = wbuf + (uint32_t)(buf * sh.unit_bytes);
#pragma unroll
        for (int rr = 0; rr < kDnRows; rr++)
#pragma unroll
            for (int k = 0; k < CPL; k++)
                if (full_lanes || lane + 32 * k < C)
                    cp_async16(dst + (uint32_t)(rr * sh.rowbytes + 512 * k), src + (size_t)rr * sh.rowbytes + 512 * k);
    };
#pragma unroll
    for (int b = 0; b < kDnBufs; b++) {
        if (q + b * nq < sh.RB) issue(q + b * nq, b);
        cp_async_commit();
    }

    // ---- wait for gate/up; this lane's chunks of slot j's h as digits --------------
    pdl_wait();
    const float hmax = __uint_as_float(__ldcg(p.ws.hmax + j));
    const float hs = hmax / kQMax;                    // NaN propagates
    const float inv = (hs > 0.0f && isfinite(hs)) ? 1.0f / hs : 0.0f;
    const float wj = (j < K) ? __ldcg(p.ws.topk_w + j) : 1.0f;
    const float coef_j = wj * hs;
    uint4 dig[CPL][6];
    int corr[3] = {0, 0, 0};
#pragma unroll
    for (int k = 0; k < CPL; k++) {
        const int c = lane + 32 * k;
        if (full_lanes || c < C) {
            const float4 *h4 = reinterpret_cast<const float4 *>(p.ws.h + (size_t)j * d.I_max + (size_t)c * 32);
            float v[32];
#pragma unroll
            for (int t = 0; t < 8; t++) {
                const float4 f = __ldcg(h4 + t);
                v[4 * t] = f.x; v[4 * t + 1] = f.y; v[4 * t + 2] = f.z; v[4 * t + 3] = f.w;
            }
            int ds[3];
            quant_chunk(v, inv, dig[k], ds);
            corr[0] -= 8 * ds[0]; corr[1] -= 8 * ds[1]; corr[2] -= 8 * ds[2];
        } else {
#pragma unroll
            for (int t = 0; t < 6; t++) dig[k][t] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    // every block has read hmax: the last one to get here clears it for the next call
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.ws.counters + 2, 1u) == gridDim.x - 1) {
            for (int jj = 0; jj < J; jj++) p.ws.hmax[jj] = 0u;
            p.ws.counters[2] = 0u;
        }
    }

    // ---- stream row blocks --------------------------------------------------------
    // lane l ends with row l / 4 of the unit
    const bool writer = (lane & 3) == 0;
    int buf = 0;
    for (int rb = q; rb < sh.RB; rb += nq, buf = (buf + 1 == kDnBufs) ? 0 : buf + 1) {
        const int o = rb * kDnRows + (lane >> 2);
        const float coef = writer ? coef_j * __ldg(sd + o) : 0.0f;   // issued before the wait
        static_assert(kDnBufs == 3, "wait_group count below assumes three buffers");
        cp_async_wait_2();
        const uint32_t st = wbuf + (uint32_t)(buf * sh.unit_bytes);
        int lo[kDnRows][3], hi[kDnRows][3];
#pragma unroll
        for (int rr = 0; rr < kDnRows; rr++) {
            lo[rr][0] = corr[0]; lo[rr][1] = corr[1]; lo[rr][2] = corr[2];
            hi[rr][0] = 0; hi[rr][1] = 0; hi[rr][2] = 0;
        }
#pragma unroll
        for (int k = 0; k < CPL; k++) {
            if (full_lanes || lane + 32 * k < C) {
#pragma unroll
                for (int rr = 0; rr < kDnRows; rr++) {
                    const uint4 w = lds128(st + (uint32_t)(rr * sh.rowbytes + 512 * k));
                    dot_chunk_lh(w, dig[k], lo[rr], hi[rr]);
                }
            }
        }
        float v[kDnRows];
#pragma unroll
        for (int rr = 0; rr < kDnRows; rr++) v[rr] = planes_lh_to_float(lo[rr], hi[rr]);
        const float tot = reduce_scatter<kDnRows>(v, lane);
        if (writer) p.ws.dpart[(size_t)j * H + o] = tot * coef;
        if (rb + kDnBufs * nq < sh.RB) issue(rb + kDnBufs * nq, buf);
        cp_async_commit();
    }
    cp_async_wait_0();
}

// y = sum_k (w_k d_k) over k ascending, then + d_shared (and + x with pre-norm
// residual); runs once the down grid has finished.
__global__ void __launch_bounds__(256) combine_decode_kernel(Params p, const float *__restrict__ x,
                                                             float *__restrict__ y) {
    pdl_wait();
    const int o = blockIdx.x * 256 + threadIdx.x;
    const Dims &d = p.d;
    if (o >= d.H) return;
    float acc = 0.0f;
    for (int k = 0; k < d.K; k++) acc += __ldcg(p.ws.dpart + (size_t)k * d.H + o);
    if (d.n_shared) acc += __ldcg(p.ws.dpart + (size_t)d.K * d.H + o);
    y[o] = d.prenorm ? x[o] + acc : acc;
}

int g_sms = 0;

constexpr int kMaxCpl = 8;     // gate/up: H up to 8192
constexpr int kMaxCplDn = 3;   // down: I up to 3072 (digits of more chunks do not fit in registers)

template <int CPL>
cudaError_t launch_gu(cudaLaunchConfig_t &cfg, const Params &p, const float *x, const GuShape &gs) {
    return cudaLaunchKernelEx(&cfg, gateup_stream_kernel<CPL>, p, x, gs);
}
template <int CPL>
cudaError_t launch_dn(cudaLaunchConfig_t &cfg, const Params &p, const DnShape &ds) {
    return cudaLaunchKernelEx(&cfg, down_stream_kernel<CPL>, p, ds);
}

cudaError_t dispatch_gu(int cpl, cudaLaunchConfig_t &cfg, const Params &p, const float *x, const GuShape &gs) {
    switch (cpl) {
        case 1: return launch_gu<1>(cfg, p, x, gs);
        case 2: return launch_gu<2>(cfg, p, x, gs);
        case 3: return launch_gu<3>(cfg, p, x, gs);
        case 4: return launch_gu<4>(cfg, p, x, gs);
        case 5: return launch_gu<5>(cfg, p, x, gs);
        case 6: return launch_gu<6>(cfg, p, x, gs);
        case 7: return launch_gu<7>(cfg, p, x, gs);
        case 8: return launch_gu<8>(cfg, p, x, gs);
    }
    return cudaErrorInvalidValue;
}
cudaError_t dispatch_dn(int cpl, cudaLaunchConfig_t &cfg, const Params &p, const DnShape &ds) {
    switch (cpl) {
        case 1: return launch_dn<1>(cfg, p, ds);
        case 2: return launch_dn<2>(cfg, p, ds);
        case 3: return launch_dn<3>(cfg, p, ds);
    }
    return cudaErrorInvalidValue;
}

template <int CPL>
cudaError_t set_smem_attr() {
    cudaError_t e = cudaFuncSetAttribute(gateup_stream_kernel<CPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGuSmemBudget);
    if (e == cudaSuccess && CPL <= kMaxCplDn)
        e = cudaFuncSetAttribute(down_stream_kernel<(CPL <= kMaxCplDn ? CPL : 1)>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kDnSmemBudget);
    return e;
}

}  // namespace

bool decode_fast_supported(const Dims &d) {
    if (d.H % kDnRows != 0 || d.H % 32 != 0 || d.I % 32 != 0 || d.I % kGuRows != 0) return false;
    if (d.n_shared && d.I_sh != d.I) return false;
    if (d.K + d.n_shared > kMaxSlots || d.K + d.n_shared > 32) return false;
    if ((d.H / 32 + 31) / 32 > kMaxCpl || (d.I / 32 + 31) / 32 > kMaxCplDn) return false;
    return gu_shape(d).smem <= (size_t)kGuSmemBudget && dn_shape(d).smem <= (size_t)kDnSmemBudget;
}

cudaError_t prepare_decode_fast(const Dims &d) {
    if (!decode_fast_supported(d)) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    // the largest any supported shape asks for, so handles of different shapes coexist
    if (e == cudaSuccess) e = set_smem_attr<1>();
    if (e == cudaSuccess) e = set_smem_attr<2>();
    if (e == cudaSuccess) e = set_smem_attr<3>();
    if (e == cudaSuccess) e = set_smem_attr<4>();
    if (e == cudaSuccess) e = set_smem_attr<5>();
    if (e == cudaSuccess) e = set_smem_attr<6>();
    if (e == cudaSuccess) e = set_smem_attr<7>();
    if (e == cudaSuccess) e = set_smem_attr<8>();
    return e;
}

// The router has been launched already (it lets these kernels start early).
// ev (optional): ev[2] after gate/up, ev[3] after down, ev[4] after the combine.
cudaError_t launch_decode_fast(const Params &p, const float *x, float *y, cudaStream_t st, cudaEvent_t *ev) {
    const GuShape gs = gu_shape(p.d);
    const DnShape ds = dn_shape(p.d);
    const int sms = g_sms > 0 ? g_sms : 148;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    const int gu_blocks = (gs.units + kWarps - 1) / kWarps;
    cfg.gridDim = dim3(gu_blocks < sms ? gu_blocks : sms);
    cfg.dynamicSmemBytes = gs.smem;
    cudaError_t e = dispatch_gu((gs.C + 31) / 32, cfg, p, x, gs);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[2], st);
    if (e != cudaSuccess) return e;

    // at least one warp per slot; otherwise one block per SM
    const int dn_units = ds.RB * ds.J;
    const int dn_blocks = (dn_units + kWarps - 1) / kWarps;
    int nb = dn_blocks < sms ? dn_blocks : sms;
    if (nb * kWarps < ds.J) nb = (ds.J + kWarps - 1) / kWarps;
    cfg.gridDim = dim3(nb);
    cfg.dynamicSmemBytes = ds.smem;
    e = dispatch_dn((ds.C + 31) / 32, cfg, p, ds);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[3], st);
    if (e != cudaSuccess) return e;

    cfg.gridDim = dim3((p.d.H + 255) / 256);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, combine_decode_kernel, p, x, y);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[4], st);
    return e;
}

}  // namespace moe
