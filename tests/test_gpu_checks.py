"""The checked build (MOE_FLAG_DEBUG_CHECKS): on every path the checks pass and
change nothing in the output, and a planted bad top-K index (written into the
workspace after a call; no step ever runs on it) makes them fail with the
failing pair recorded, after which the handle recovers."""
import pytest

import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import int4_moe_expert_gb300 as m
    return m


def _layer(moe, wl, li, max_tokens, **kw):
    cfg = moe.make_config(wl.H, wl.E, wl.K, wl.I, wl.n_shared, wl.I_shared, wl.routed_scale,
                          wl.norm_topk, wl.prenorm_residual, wl.rms_eps, n_group=wl.n_group,
                          topk_group=wl.topk_group, score_func=wl.score_func,
                          expert_format=wl.expert_format, shared_format=wl.shared_format, **kw)
    rows = None
    if cfg.ep_size > 1:
        from int4_moe_expert_gb300.expert_parallel import owned_range
        lo, hi = owned_range(wl.E, cfg.ep_size, cfg.ep_rank)
        rows = [e if lo <= e < hi else None for e in range(wl.E)]
    shared = cfg.n_shared and cfg.ep_rank == 0
    return moe.MoeLayer(cfg, li.router_w, li.router_b, li.slabs, li.scales,
                        li.sh_slab if shared else None, li.sh_scale if shared else None,
                        max_tokens=max_tokens, expert_rows=rows)


CASES = [
    ("tiny", 1, {}),                      # single-kernel decode
    ("group8", 1, {}),                    # single-kernel decode, routing variant
    ("olmoe_int8", 1, {}),                # single-kernel decode, int8
    ("olmoe", 5, {}),                     # mma.sync experts, buckets
    ("olmoe", 300, {}),                   # tcgen05 experts
    ("g64_35b", 1, {}),                   # tensor-core experts at T = 1 (group-64)
    ("tiny", 37, {"cuda_cores": True}),   # CUDA-core batched kernels
    ("olmoe", 5, {"ep_size": 2, "ep_rank": 1}),   # expert parallelism: other rank's pairs
    ("stack35b", 1, {"ep_size": 3, "ep_rank": 0}),
]


@pytest.mark.parametrize("name,T,kw", CASES)
def test_checks_pass_and_change_nothing(moe, name, T, kw):
    wl = synth.WORKLOADS[name]
    li = synth.layer_inputs(wl)
    x = torch.from_numpy(synth.tokens(wl, T=T, stream=5)).cuda()
    plain = _layer(moe, wl, li, T, **kw)
    checked = _layer(moe, wl, li, T, debug_checks=True, **kw)
    try:
        a, ia, wa = plain.forward_debug(x)
        b, ib, wb = checked.forward_debug(x)
        assert moe.moe_device_error(checked.handle, check=False) == 0
        assert moe.moe_debug_check_result(checked.handle) == (-1, 0)
        assert torch.equal(a, b) and torch.equal(ia, ib) and torch.equal(wa, wb)
    finally:
        plain.close()
        checked.close()


@pytest.mark.parametrize("name,T", [("olmoe", 5), ("tiny", 1)])
def test_planted_index_is_caught(moe, name, T):
    wl = synth.WORKLOADS[name]
    li = synth.layer_inputs(wl)
    layer = _layer(moe, wl, li, T)
    x = torch.from_numpy(synth.tokens(wl, T=T, stream=6)).cuda()
    try:
        _, idx, _ = layer.forward_debug(x)
        idx = idx.cpu().numpy().ravel()
        moe.moe_debug_check(layer.handle, T)
        assert moe.moe_debug_check_result(layer.handle) == (-1, 0)
        assert moe.moe_device_error(layer.handle, check=False) == 0
        K, P = wl.K, T * wl.K
        plants = [(min(3, P - 1), wl.E + 5, {1, 6, 7}),   # out of range (and, with buckets, the totals)
                  (min(3, P - 1), -1, {1, 6, 7}),
                  (1, int(idx[0]), {3, 5, 6})]             # repeats the token's first choice
        for pair, val, codes in plants:
            moe.moe_debug_set_topk(layer.handle, pair, val)
            moe.moe_debug_check(layer.handle, T)
            where, code = moe.moe_debug_check_result(layer.handle)
            assert code in codes, (pair, val, where, code)
            assert where == pair or where >= P, (pair, where)
            f = moe.moe_device_error(layer.handle, check=False)
            assert f & moe.MOE_DEVICE_ERR_CHECK
            assert moe.moe_debug_check_result(layer.handle) == (-1, 0)   # cleared by the reset
            moe.moe_debug_set_topk(layer.handle, pair, int(idx[pair]))   # restore
        # a fresh call rewrites the routing; its checks pass again
        layer.forward_debug(x)
        moe.moe_debug_check(layer.handle, T)
        assert moe.moe_debug_check_result(layer.handle) == (-1, 0)
        assert moe.moe_device_error(layer.handle, check=False) == 0
    finally:
        layer.close()
