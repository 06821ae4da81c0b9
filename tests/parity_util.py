"""Helpers shared by the GPU parity tests: upload a synthetic layer, compare a
GPU call with the oracle under the selection-margin rule."""
from __future__ import annotations

import numpy as np

import oracle
import synth

MARGIN = 1e-5      # selection must match exactly when c_(K) - c_(K+1) > MARGIN
REL_TOL = 2e-3     # per token: max|y - y_ref| / max|y_ref|
W_RTOL = 1e-4      # routing weights, per expert id (float32 sigmoid vs double)


def gpu_config(moe, wl):
    return moe.make_config(wl.H, wl.E, wl.K, wl.I, wl.n_shared, wl.I_shared, wl.routed_scale,
                           wl.norm_topk, wl.prenorm_residual, wl.rms_eps, n_group=wl.n_group,
                           topk_group=wl.topk_group, score_func=wl.score_func,
                           expert_format=wl.expert_format, shared_format=wl.shared_format)


def upload(moe, wl, li, max_tokens):
    return moe.MoeLayer(gpu_config(moe, wl), li.router_w, li.router_b, li.slabs, li.scales,
                        li.sh_slab, li.sh_scale, max_tokens=max_tokens)


def oracle_layer(wl, li, experts=None):
    return oracle.LayerRef.from_inputs(oracle.cfg_from_workload(wl), li, experts)


def rel_err(y, y_ref):
    den = np.abs(y_ref).max()
    return float(np.abs(y - y_ref).max() / (den if den > 0 else 1.0))


def elem_err(y, y_ref):
    """Element-wise diagnostic beside the per-token bar: max over elements of
    |y - y_ref| / max(|y_ref|, 1e-3 rms(y_ref)), so that small outputs are
    looked at one by one (reported, not asserted)."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    floor = 1e-3 * float(np.sqrt(np.mean(y_ref * y_ref)))
    den = np.maximum(np.abs(y_ref), floor if floor > 0 else 1e-300)
    return float(np.max(np.abs(np.asarray(y, dtype=np.float64) - y_ref) / den))


# worst per-token and element-wise errors seen per test, printed at the end of the run
DIAG = {}


def record(where: str, err: float, eerr: float) -> None:
    key = where.split(" t=")[0]
    a, b = DIAG.get(key, (0.0, 0.0))
    DIAG[key] = (max(a, err), max(b, eerr))


def check_route(wl, cfg, router_w, router_b, x_in, idx_gpu, w_gpu, where=""):
    """Check one token's routing decision against the oracle (x_in: the router
    input, pre-normed where the layer asks for it).  Returns (forced, near_tie):
    forced is the GPU's selection when the oracle's own is within the margin
    (the output must then be checked with that selection), else None."""
    idx_ref, w_ref, margin, scores = oracle.route(cfg, router_w, router_b, x_in)
    choice = scores[2]
    idx_gpu = np.asarray(idx_gpu, dtype=np.int64)
    assert np.all((idx_gpu >= 0) & (idx_gpu < wl.E)), (where, idx_gpu)
    assert len(set(idx_gpu.tolist())) == wl.K, (where, idx_gpu)
    near_tie = margin <= MARGIN
    if not near_tie:
        assert sorted(idx_gpu.tolist()) == sorted(idx_ref.tolist()), (where, idx_gpu, idx_ref, margin)
        forced = None
    else:
        if wl.n_group > 1:
            # a near-tie may be between two groups: the GPU's set is then checked through
            # the output recomputed with it (its experts may lie in a group the oracle dropped)
            in_kept = np.isfinite(choice[idx_gpu])
            choice = np.where(np.isfinite(choice), choice, scores[1] + np.asarray(router_b, np.float64))
            assert in_kept.any(), (where, idx_gpu)
        kth = choice[idx_ref[-1]]
        if wl.n_group == 1:
            assert np.all(choice[idx_gpu] >= kth - MARGIN), (where, idx_gpu, idx_ref, margin)
        forced = idx_gpu.astype(np.int32)
    # GPU order is descending selection score (up to float32 rounding)
    c = choice[idx_gpu]
    assert np.all(c[:-1] >= c[1:] - MARGIN), (where, c)
    # weights compared per expert id, against the oracle's weights of the GPU's own set
    w_used = w_ref if forced is None else oracle.weights_for(cfg, router_w, x_in, forced)
    idx_used = idx_ref if forced is None else forced
    ref_w = dict(zip(np.asarray(idx_used).tolist(), np.asarray(w_used).tolist()))
    for e, w in zip(idx_gpu.tolist(), np.asarray(w_gpu, dtype=np.float64).tolist()):
        assert abs(w - ref_w[e]) <= W_RTOL * max(abs(ref_w[e]), 1e-30), (where, e, w, ref_w[e])
    return forced, near_tie


def check_token(wl, ref: oracle.LayerRef, x_t, y_gpu, idx_gpu, w_gpu, where=""):
    """Check one token.  Returns (rel_err, near_tie)."""
    x64 = np.asarray(x_t, dtype=np.float64)
    xin = oracle.rmsnorm(x64, wl.rms_eps) if wl.prenorm_residual else x64
    forced, near_tie = check_route(wl, ref.cfg, ref.router_w, ref.router_b, xin, idx_gpu, w_gpu, where)
    y_ref, _, _, _ = ref.token(x64, forced_idx=forced)
    y64 = np.asarray(y_gpu, dtype=np.float64)
    err = rel_err(y64, y_ref)
    record(where, err, elem_err(y64, y_ref))
    assert err <= REL_TOL, (where, err)
    return err, near_tie


def selected_experts(wl, li, x, experts_hint=None):
    """Experts the oracle needs for these tokens (its own choice plus any hint)."""
    ref = oracle_layer(wl, li, experts=[])
    need = set(experts_hint or [])
    for t in range(x.shape[0]):
        x64 = x[t].astype(np.float64)
        xin = oracle.rmsnorm(x64, wl.rms_eps) if wl.prenorm_residual else x64
        idx, _, _, _ = oracle.route(ref.cfg, ref.router_w, ref.router_b, xin)
        need.update(idx.tolist())
    return need


def oracle_ep_partial(wl, li, x_t, lo: int, hi: int, rank0: bool, idx=None):
    """One expert-parallel rank's partial output of token x_t, in double: the
    selected experts with lo <= e < hi (routing weights over the whole
    selection), plus the shared expert and the pre-norm residual on rank 0.
    idx: a selection to use instead of the oracle's own (near-ties)."""
    cfg = oracle.cfg_from_workload(wl)
    x64 = np.asarray(x_t, dtype=np.float64)
    xin = oracle.rmsnorm(x64, wl.rms_eps) if wl.prenorm_residual else x64
    if idx is None:
        idx, w, _, _ = oracle.route(cfg, li.router_w, li.router_b, xin)
    else:
        w = oracle.weights_for(cfg, li.router_w, xin, idx)
    y = np.zeros(wl.H, dtype=np.float64)
    for e, we in zip(np.asarray(idx).tolist(), np.asarray(w).tolist()):
        if lo <= e < hi:
            d, _ = oracle.expert(wl.H, wl.I, li.slabs[e], li.scales[e], xin, wl.expert_format)
            y += we * d
    if rank0:
        if wl.n_shared:
            d, _ = oracle.expert(wl.H, wl.I_shared, li.sh_slab, li.sh_scale, xin, wl.shared_format)
            y += d
        if wl.prenorm_residual:
            y += x64
    return y
