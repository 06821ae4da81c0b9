// C-ABI layer of the int4 routed-MoE FFN library: argument validation,
// workspace ownership, error reporting.  All compute is in moe_kernels.cu.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>

#include "moe_internal.h"

struct moe_handle {
    moe::Params p;
    void *ws_base;
    size_t ws_bytes;
    void *tables;        // device copies of the per-expert pointer arrays
    void *tmaps;         // tcgen05 path: tensor maps of the weights and activations (or NULL)
    float *x_stage;      // device staging for moe_forward_host
    float *y_stage;
    int device;
    cudaEvent_t *prof_ev;   // [prof_max][kStages + 1]
    int prof_max;           // calls to record
    int prof_n;             // calls recorded so far
    int last_T;             // tokens of the last call, and whether it built buckets (checks)
    bool last_buckets;
};

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

moe_status cuda_fail(cudaError_t e, const char *what) {
    const moe_status s = (e == cudaErrorMemoryAllocation) ? MOE_ERR_NOMEM : MOE_ERR_CUDA;
    return fail(s, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

constexpr int kMaxTokens = 1 << 16;

moe_status check_config(const moe_config *c, int32_t max_tokens, moe::Dims *d) {
    if (!c) return fail(MOE_ERR_INVALID, "config is NULL");
    if (c->hidden < 32 || c->hidden > 16384 || c->hidden % 32)
        return fail(MOE_ERR_UNSUPPORTED, "hidden=%d: need a multiple of 32 in [32, 16384]", c->hidden);
    if (c->n_experts < 1 || c->n_experts > 1024)
        return fail(MOE_ERR_UNSUPPORTED, "n_experts=%d: need 1..1024", c->n_experts);
    if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > 32)
        return fail(MOE_ERR_INVALID, "top_k=%d: need 1..min(n_experts, 32)", c->top_k);
    if (c->moe_inter < 32 || c->moe_inter > 16384 || c->moe_inter % 32)
        return fail(MOE_ERR_UNSUPPORTED, "moe_inter=%d: need a multiple of 32 in [32, 16384]", c->moe_inter);
    if (c->n_shared != 0 && c->n_shared != 1)
        return fail(MOE_ERR_UNSUPPORTED, "n_shared=%d: need 0 or 1", c->n_shared);
    if (c->n_shared == 1 &&
        (c->shared_inter < 32 || c->shared_inter > 16384 || c->shared_inter % 32))
        return fail(MOE_ERR_UNSUPPORTED, "shared_inter=%d: need a multiple of 32 in [32, 16384]",
                    c->shared_inter);
    if (c->expert_format < MOE_FORMAT_INT4 || c->expert_format > MOE_FORMAT_G64 ||
        c->shared_format < MOE_FORMAT_INT4 || c->shared_format > MOE_FORMAT_G64)
        return fail(MOE_ERR_INVALID, "expert_format / shared_format: need a MOE_FORMAT_* value");
    if (c->expert_format != MOE_FORMAT_INT4 || (c->n_shared && c->shared_format != MOE_FORMAT_INT4)) {
        if (c->hidden % 128 || c->moe_inter % 128 || (c->n_shared && c->shared_inter % 128))
            return fail(MOE_ERR_UNSUPPORTED, "int8 / group-64 experts need H, I and I_shared multiples of 128");
        if (c->flags & MOE_FLAG_CUDA_CORES)
            return fail(MOE_ERR_UNSUPPORTED, "int8 / group-64 experts run on the tensor-core kernels only");
    }
    if (c->score_func != MOE_SCORE_SIGMOID && c->score_func != MOE_SCORE_SOFTMAX)
        return fail(MOE_ERR_INVALID, "score_func=%d: need MOE_SCORE_SIGMOID or MOE_SCORE_SOFTMAX", c->score_func);
    if (c->n_group < 1 || c->n_group > 32 || c->n_experts % c->n_group)
        return fail(MOE_ERR_INVALID, "n_group=%d: need 1..32 dividing n_experts", c->n_group);
    if (c->n_group > 1) {
        if (c->score_func != MOE_SCORE_SIGMOID)
            return fail(MOE_ERR_INVALID, "n_group > 1 needs the sigmoid score");
        if (c->topk_group < 1 || c->topk_group > c->n_group)
            return fail(MOE_ERR_INVALID, "topk_group=%d: need 1..n_group", c->topk_group);
        if (c->top_k > c->topk_group * (c->n_experts / c->n_group))
            return fail(MOE_ERR_INVALID, "top_k=%d exceeds the experts of the kept groups", c->top_k);
    }
    if (c->norm_topk != 0 && c->norm_topk != 1)
        return fail(MOE_ERR_INVALID, "norm_topk=%d: need 0 or 1", c->norm_topk);
    if (!isfinite(c->routed_scale)) return fail(MOE_ERR_INVALID, "routed_scale is not finite");
    if (c->flags & ~(MOE_FLAG_PRENORM_RESIDUAL | MOE_FLAG_TRACE | MOE_FLAG_CUDA_CORES | MOE_FLAG_DEBUG_CHECKS))
        return fail(MOE_ERR_INVALID, "unknown flags 0x%x", c->flags);
    if ((c->flags & MOE_FLAG_PRENORM_RESIDUAL) && !(c->rms_eps >= 0.0f && isfinite(c->rms_eps)))
        return fail(MOE_ERR_INVALID, "rms_eps must be finite and >= 0");
    if (max_tokens < 1 || max_tokens > kMaxTokens)
        return fail(MOE_ERR_INVALID, "max_tokens=%d: need 1..%d", max_tokens, kMaxTokens);
    const int ep = c->ep_size == 0 ? 1 : c->ep_size;
    if (ep < 1 || ep > c->n_experts || c->ep_rank < 0 || c->ep_rank >= ep)
        return fail(MOE_ERR_INVALID, "ep_size=%d, ep_rank=%d: need 1 <= ep_size <= n_experts, 0 <= ep_rank < ep_size",
                    c->ep_size, c->ep_rank);
    d->H = c->hidden;
    d->E = c->n_experts;
    d->K = c->top_k;
    d->I = c->moe_inter;
    d->n_shared = (c->n_shared && c->ep_rank == 0) ? 1 : 0;   // the shared expert is rank 0's
    d->I_sh = d->n_shared ? c->shared_inter : 0;
    d->I_max = d->I > d->I_sh ? d->I : d->I_sh;
    d->norm_topk = c->norm_topk;
    d->n_group = c->n_group;
    d->topk_group = c->n_group > 1 ? c->topk_group : 1;
    d->score_func = c->score_func;
    d->expert_fmt = c->expert_format;
    d->shared_fmt = d->n_shared ? c->shared_format : MOE_FORMAT_INT4;
    d->mma_fmt = (d->expert_fmt != MOE_FORMAT_INT4 || d->shared_fmt != MOE_FORMAT_INT4) ? 1 : 0;
    d->tc = moe::tc_supported(*d) ? 1 : 0;
    d->prenorm = (c->flags & MOE_FLAG_PRENORM_RESIDUAL) ? 1 : 0;
    d->ep_lo = (int)((long long)c->ep_rank * c->n_experts / ep);
    d->ep_hi = (int)((long long)(c->ep_rank + 1) * c->n_experts / ep);
    d->resid = (d->prenorm && c->ep_rank == 0) ? 1 : 0;
    d->scale = c->routed_scale;
    d->eps = c->rms_eps;
    d->max_tokens = max_tokens;
    d->fast_decode = (ep == 1 && moe::decode_fast_supported(*d)) ? 1 : 0;
    d->mma = (moe::mma_supported(*d) && !(c->flags & MOE_FLAG_CUDA_CORES)) ? 1 : 0;
    d->trace = (c->flags & MOE_FLAG_TRACE) ? 1 : 0;
    d->debug_checks = (c->flags & MOE_FLAG_DEBUG_CHECKS) ? 1 : 0;
    return MOE_OK;
}

bool is_device_ptr(const void *ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

moe_status check_weights(const moe::Dims &d, const moe_weights *w) {
    if (!w) return fail(MOE_ERR_INVALID, "weights is NULL");
    if (!w->router_w || !w->router_bias) return fail(MOE_ERR_INVALID, "router_w / router_bias is NULL");
    if (!aligned16(w->router_w)) return fail(MOE_ERR_INVALID, "router_w must be 16-byte aligned");
    if (!is_device_ptr(w->router_w) || !is_device_ptr(w->router_bias))
        return fail(MOE_ERR_INVALID, "router_w / router_bias are not device pointers");
    if (!w->expert_slab || !w->expert_scale) return fail(MOE_ERR_INVALID, "expert pointer arrays are NULL");
    for (int e = d.ep_lo; e < d.ep_hi; e++) {     // the experts this handle computes
        const void *s = w->expert_slab[e], *c = w->expert_scale[e];
        if (!s || !c) return fail(MOE_ERR_INVALID, "expert %d: NULL slab or scale", e);
        if (!aligned16(s) || !aligned16(c))
            return fail(MOE_ERR_INVALID, "expert %d: slab and scale must be 16-byte aligned", e);
        if (!is_device_ptr(s) || !is_device_ptr(c))
            return fail(MOE_ERR_INVALID, "expert %d: slab / scale are not device pointers", e);
    }
    if (d.n_shared) {
        if (!w->shared_slab || !w->shared_scale) return fail(MOE_ERR_INVALID, "shared expert pointers are NULL");
        if (!aligned16(w->shared_slab) || !aligned16(w->shared_scale))
            return fail(MOE_ERR_INVALID, "shared slab and scale must be 16-byte aligned");
        if (!is_device_ptr(w->shared_slab) || !is_device_ptr(w->shared_scale))
            return fail(MOE_ERR_INVALID, "shared slab / scale are not device pointers");
    }
    return MOE_OK;
}

void free_events(moe_handle *h) {
    if (h->prof_ev) {
        for (int i = 0; i < h->prof_max * (moe::kStages + 1); i++)
            if (h->prof_ev[i]) cudaEventDestroy(h->prof_ev[i]);
        delete[] h->prof_ev;
    }
    h->prof_ev = nullptr;
    h->prof_max = 0;
    h->prof_n = 0;
}

void free_handle(moe_handle *h) {
    if (!h) return;
    free_events(h);
    if (h->ws_base) cudaFree(h->ws_base);
    if (h->tables) cudaFree(h->tables);
    if (h->tmaps) cudaFree(h->tmaps);
    if (h->x_stage) cudaFree(h->x_stage);
    if (h->y_stage) cudaFree(h->y_stage);
    delete h;
}

bool ranges_overlap(const void *a, const void *b, size_t n) {
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + n && pb < pa + n;
}

moe_status run(moe_handle *h, const float *x, int32_t T, float *y, int32_t *topk_idx,
               float *topk_w, int32_t *counts, void *stream, bool debug) {
    if (!h) return fail(MOE_ERR_INVALID, "handle is NULL");
    if (T < 0 || T > h->p.d.max_tokens)
        return fail(MOE_ERR_INVALID, "T=%d: need 0..max_tokens=%d", T, h->p.d.max_tokens);
    if (T == 0) return MOE_OK;
    if (!x || !y) return fail(MOE_ERR_INVALID, "x / y is NULL");
    if (!aligned16(x) || !aligned16(y)) return fail(MOE_ERR_INVALID, "x and y must be 16-byte aligned");
    const size_t bytes = (size_t)T * h->p.d.H * sizeof(float);
    if (ranges_overlap(x, y, bytes)) return fail(MOE_ERR_INVALID, "x and y overlap");
    if (debug && (!topk_idx || !topk_w)) return fail(MOE_ERR_INVALID, "topk_idx / topk_w is NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device)
        return fail(MOE_ERR_INVALID, "current device %d is not the handle's device %d", dev, h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t *ev = nullptr;
    if (h->prof_ev && h->prof_n < h->prof_max) ev = h->prof_ev + (size_t)(h->prof_n++) * (moe::kStages + 1);
    e = moe::launch_forward(h->p, x, T, y, st, counts != nullptr, ev);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    h->last_T = T;
    h->last_buckets = moe::buckets_built(h->p.d, T, counts != nullptr);
    if (h->p.d.debug_checks) {
        e = moe::launch_checks(h->p, T, h->last_buckets, st);
        if (e != cudaSuccess) return cuda_fail(e, "check kernel launch");
    }
    if (debug) {
        const size_t nk = (size_t)T * h->p.d.K;
        e = cudaMemcpyAsync(topk_idx, h->p.ws.topk_idx, nk * sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(topk_w, h->p.ws.topk_w, nk * sizeof(float), cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && counts)
            e = cudaMemcpyAsync(counts, h->p.ws.cnt, (size_t)h->p.d.E * sizeof(int32_t),
                                cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "debug copy");
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_last_error(void) { return g_err; }

size_t moe_workspace_bytes(const moe_config *cfg, int32_t max_tokens) {
    moe::Dims d;
    if (check_config(cfg, max_tokens, &d) != MOE_OK) return 0;
    return moe::workspace_bytes(d);
}

moe_status moe_init(const moe_config *cfg, const moe_weights *w, int32_t max_tokens, moe_handle **out) {
    if (!out) return fail(MOE_ERR_INVALID, "out is NULL");
    *out = nullptr;
    g_err[0] = '\0';
    moe::Dims d;
    moe_status s = check_config(cfg, max_tokens, &d);
    if (s != MOE_OK) return s;
    s = check_weights(d, w);
    if (s != MOE_OK) return s;

    moe_handle *h = new (std::nothrow) moe_handle();
    if (!h) return fail(MOE_ERR_NOMEM, "host allocation failed");
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) { free_handle(h); return cuda_fail(e, "cudaGetDevice"); }

    h->ws_bytes = moe::workspace_bytes(d);
    e = cudaMalloc(&h->ws_base, h->ws_bytes);
    if (e != cudaSuccess) { h->ws_base = nullptr; free_handle(h); return cuda_fail(e, "workspace cudaMalloc"); }
    const size_t tbytes = 2 * (size_t)d.E * sizeof(void *);
    e = cudaMalloc(&h->tables, tbytes);
    if (e != cudaSuccess) { h->tables = nullptr; free_handle(h); return cuda_fail(e, "table cudaMalloc"); }
    const size_t stage = (size_t)max_tokens * d.H * sizeof(float);
    e = cudaMalloc(reinterpret_cast<void **>(&h->x_stage), stage);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&h->y_stage), stage);
    if (e != cudaSuccess) { free_handle(h); return cuda_fail(e, "staging cudaMalloc"); }

    void **host_tab = new (std::nothrow) void *[2 * (size_t)d.E];
    if (!host_tab) { free_handle(h); return fail(MOE_ERR_NOMEM, "host allocation failed"); }
    for (int i = 0; i < d.E; i++) {      // experts another rank computes: NULL (never read)
        const bool own = i >= d.ep_lo && i < d.ep_hi;
        host_tab[i] = own ? const_cast<uint8_t *>(w->expert_slab[i]) : nullptr;
        host_tab[d.E + i] = own ? const_cast<float *>(w->expert_scale[i]) : nullptr;
    }
    e = cudaMemcpy(h->tables, host_tab, tbytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) { delete[] host_tab; free_handle(h); return cuda_fail(e, "table upload"); }

    moe::Params &p = h->p;
    p.d = d;
    p.router_w = w->router_w;
    p.router_b = w->router_bias;
    p.slabs = static_cast<const uint8_t *const *>(h->tables);
    p.scales = reinterpret_cast<const float *const *>(static_cast<void **>(h->tables) + d.E);
    p.sh_slab = d.n_shared ? w->shared_slab : nullptr;
    p.sh_scale = d.n_shared ? w->shared_scale : nullptr;
    moe::carve_workspace(d, h->ws_base, &p.ws);
    const size_t nmaps = moe::tc_map_count(d);
    if (nmaps) {
        e = cudaMalloc(&h->tmaps, nmaps * moe::kTmapBytes);
        if (e != cudaSuccess) { h->tmaps = nullptr; delete[] host_tab; free_handle(h); return cuda_fail(e, "tensor-map cudaMalloc"); }
        p.tmaps = h->tmaps;
        e = moe::upload_tc_maps(p, reinterpret_cast<const uint8_t *const *>(host_tab), h->tmaps);
        if (e != cudaSuccess) { delete[] host_tab; free_handle(h); return cuda_fail(e, "tensor-map encoding"); }
    } else {
        p.tmaps = nullptr;
    }
    delete[] host_tab;
    e = cudaMemset(h->ws_base, 0, h->ws_bytes);
    if (e == cudaSuccess) e = moe::prepare_kernels(p.d);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { free_handle(h); return cuda_fail(e, "workspace init"); }
    *out = h;
    return MOE_OK;
}

moe_status moe_forward(moe_handle *h, const float *x, int32_t T, float *y, void *stream) {
    return run(h, x, T, y, nullptr, nullptr, nullptr, stream, false);
}

moe_status moe_forward_debug(moe_handle *h, const float *x, int32_t T, float *y, int32_t *topk_idx,
                             float *topk_w, int32_t *expert_counts, void *stream) {
    return run(h, x, T, y, topk_idx, topk_w, expert_counts, stream, true);
}

moe_status moe_forward_host(moe_handle *h, const float *x_host, int32_t T, float *y_host, void *stream) {
    if (!h) return fail(MOE_ERR_INVALID, "handle is NULL");
    if (T < 0 || T > h->p.d.max_tokens)
        return fail(MOE_ERR_INVALID, "T=%d: need 0..max_tokens=%d", T, h->p.d.max_tokens);
    if (T == 0) return MOE_OK;
    if (!x_host || !y_host) return fail(MOE_ERR_INVALID, "x_host / y_host is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)T * h->p.d.H * sizeof(float);
    cudaError_t e = cudaMemcpyAsync(h->x_stage, x_host, bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "input copy");
    moe_status s = run(h, h->x_stage, T, h->y_stage, nullptr, nullptr, nullptr, stream, false);
    if (s != MOE_OK) return s;
    e = cudaMemcpyAsync(y_host, h->y_stage, bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "output copy");
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    return MOE_OK;
}

moe_status moe_profile_start(moe_handle *h, int32_t max_calls) {
    if (!h) return fail(MOE_ERR_INVALID, "handle is NULL");
    if (max_calls < 0 || max_calls > 4096) return fail(MOE_ERR_INVALID, "max_calls=%d: need 0..4096", max_calls);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
    free_events(h);
    if (max_calls == 0) return MOE_OK;
    const int n = max_calls * (moe::kStages + 1);
    h->prof_ev = new (std::nothrow) cudaEvent_t[n]();
    if (!h->prof_ev) return fail(MOE_ERR_NOMEM, "host allocation failed");
    h->prof_max = max_calls;
    for (int i = 0; i < n; i++) {
        e = cudaEventCreate(&h->prof_ev[i]);
        if (e != cudaSuccess) { free_events(h); return cuda_fail(e, "cudaEventCreate"); }
    }
    return MOE_OK;
}

moe_status moe_profile_read(moe_handle *h, int32_t *n_calls, float *stage_ms) {
    if (!h || !n_calls || !stage_ms) return fail(MOE_ERR_INVALID, "NULL argument");
    *n_calls = h->prof_n;
    for (int s = 0; s < moe::kStages; s++) stage_ms[s] = 0.0f;
    if (!h->prof_ev || h->prof_n == 0) return MOE_OK;
    double sum[moe::kStages] = {0, 0, 0, 0};
    for (int c = 0; c < h->prof_n; c++) {
        cudaEvent_t *ev = h->prof_ev + (size_t)c * (moe::kStages + 1);
        cudaError_t e = cudaEventSynchronize(ev[moe::kStages]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
        for (int s = 0; s < moe::kStages; s++) {
            float ms = 0.0f;
            e = cudaEventElapsedTime(&ms, ev[s], ev[s + 1]);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
            sum[s] += ms;
        }
    }
    for (int s = 0; s < moe::kStages; s++) stage_ms[s] = (float)(sum[s] / h->prof_n);
    return MOE_OK;
}

moe_status moe_device_error(moe_handle *h, uint32_t *flags) {
    if (!h || !flags) return fail(MOE_ERR_INVALID, "NULL argument");
    unsigned v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, h->p.ws.err, sizeof(v), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && v) {
        // a kernel gave up part-way: start the barrier counters and the call
        // counter afresh so that the next call is consistent again (until this
        // reset, every call on the handle is invalid)
        e = cudaMemset(h->p.ws.counters, 0, 16 * sizeof(unsigned));
        if (e == cudaSuccess) e = cudaMemset(h->p.ws.err, 0, 4 * sizeof(unsigned));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
    }
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    *flags = v;
    if (v) return fail(MOE_ERR_CUDA, "a kernel gave up waiting (flags 0x%x)", v);
    return MOE_OK;
}

moe_status moe_debug_check(moe_handle *h, int32_t T) {
    if (!h) return fail(MOE_ERR_INVALID, "handle is NULL");
    if (T < 1 || T > h->p.d.max_tokens) return fail(MOE_ERR_INVALID, "T=%d: need 1..max_tokens", T);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = moe::launch_checks(h->p, T, T == h->last_T && h->last_buckets, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "check kernel");
    return MOE_OK;
}

moe_status moe_debug_set_topk(moe_handle *h, int32_t pair, int32_t expert) {
    if (!h) return fail(MOE_ERR_INVALID, "handle is NULL");
    if (pair < 0 || (long long)pair >= (long long)h->p.d.max_tokens * h->p.d.K)
        return fail(MOE_ERR_INVALID, "pair=%d: need 0..max_tokens*K-1", pair);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(h->p.ws.topk_idx + pair, &expert, sizeof(expert), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "writing the top-K index");
    return MOE_OK;
}

moe_status moe_debug_check_result(moe_handle *h, int32_t *pair, int32_t *code) {
    if (!h || !pair || !code) return fail(MOE_ERR_INVALID, "NULL argument");
    unsigned v[4] = {0, 0, 0, 0};
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(v, h->p.ws.err, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the check record");
    *pair = v[1] ? (int32_t)(v[1] - 1) : -1;
    *code = v[1] ? (int32_t)v[2] : 0;
    return MOE_OK;
}

moe_status moe_debug_stall_next_call(moe_handle *h) {
    if (!h) return fail(MOE_ERR_INVALID, "handle is NULL");
    if (!h->p.d.fast_decode) return fail(MOE_ERR_UNSUPPORTED, "T == 1 calls on this handle do not use the decode kernel");
    // counters[7] is the number of the handle's last call; every barrier target of the next
    // call is that number + 1 times the grid, which the barrier counters (at most the calls
    // so far times the grid) then cannot reach
    unsigned calls = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&calls, h->p.ws.counters + 7, sizeof(calls), cudaMemcpyDeviceToHost);
    calls += 1000u;
    if (e == cudaSuccess) e = cudaMemcpy(h->p.ws.counters + 7, &calls, sizeof(calls), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "moving the call counter");
    return MOE_OK;
}

int32_t moe_uses_streaming_decode(const moe_handle *h) { return h ? h->p.d.fast_decode : 0; }

int32_t moe_streaming_decode_max_tokens(const moe_handle *h) {
    return (h && h->p.d.fast_decode) ? moe::decode_loop_max_tokens() : 0;
}

int32_t moe_uses_tensor_cores(const moe_handle *h) { return h ? h->p.d.mma : 0; }

moe_status moe_trace_read(moe_handle *h, uint64_t *out, int32_t capacity_blocks, int32_t *n_blocks) {
    if (!h || !out || !n_blocks || capacity_blocks < 0) return fail(MOE_ERR_INVALID, "NULL argument or negative capacity");
    if (!h->p.d.trace || !h->p.d.fast_decode)
        return fail(MOE_ERR_UNSUPPORTED, "the handle records no trace (MOE_FLAG_TRACE and the decode kernel needed)");
    const int g = moe::decode_grid_blocks(h->p.d);
    const int n = g < capacity_blocks ? g : capacity_blocks;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess && n > 0)
        e = cudaMemcpy(out, h->p.ws.trace, (size_t)n * MOE_TRACE_SLOTS * sizeof(uint64_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the trace");
    *n_blocks = g;
    return MOE_OK;
}

moe_status moe_destroy(moe_handle *h) {
    if (!h) return MOE_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    const int dev = h->device;
    if (cur != dev) cudaSetDevice(dev);
    const cudaError_t e = cudaDeviceSynchronize();
    free_handle(h);
    if (cur >= 0 && cur != dev) cudaSetDevice(cur);
    if (e != cudaSuccess) return cuda_fail(e, "device synchronize before free");
    return MOE_OK;
}

}  // extern "C"
