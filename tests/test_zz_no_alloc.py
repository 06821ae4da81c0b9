"""The allocation-free router entry point, moe_route_noalloc.

It exists for callers that may not allocate device memory (their device
memory belongs to another allocator, or their serving loop must never call
cudaMalloc/cudaFree), so it cannot use a moe_handle.  Here it is called
through the C ABI and its top-k indices and weights are compared with those
moe_forward_debug returns for the same tokens, on two calls in a row (the
static scratch keeps the previous call's contents), and with the oracle's
routing under the selection-margin rule, for the plain sigmoid router and
the group-limited and softmax variants it also accepts.  This file sorts
last so that a run stopping at the first failure has run every other test
first.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_util import W_RTOL, check_route, oracle_layer, upload

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


CASES = [
    synth.WORKLOADS["tiny"],
    synth.WORKLOADS["olmoe"],
    synth.Workload("wide", T=1, H=96, E=300, K=32, I=32, n_shared=1, I_shared=64,
                   routed_scale=2.5, seed=21),
    synth.Workload("prenorm", T=1, H=64, E=8, K=2, I=32, n_shared=1, I_shared=32,
                   routed_scale=1.0, seed=22, n_layers=2),
    synth.WORKLOADS["group8"],
    synth.WORKLOADS["softmax_renorm"],
    synth.WORKLOADS["olmoe_softmax"],
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_route_noalloc_matches_forward_debug(moe, wl):
    li = synth.layer_inputs(wl)
    layer = upload(moe, wl, li, 8)
    for call, T in enumerate((1, 8)):          # two calls in a row
        x = torch.from_numpy(synth.tokens(wl, T=T, stream=50 + call)).cuda()
        _, idx_ref, w_ref = layer.forward_debug(x)
        idx = torch.full((T, wl.K), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, wl.K), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_route_noalloc(layer.cfg, layer.router_w, layer.router_b, x, T, idx, w)
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref), (wl.name, call)
        np.testing.assert_allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=W_RTOL, atol=0)
        # and against the oracle's routing of the same tokens
        ref = oracle_layer(wl, li, experts=[])
        xh, ih, wh = x.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
        for t in range(T):
            x64 = xh[t].astype(np.float64)
            xin = oracle.rmsnorm(x64, wl.rms_eps) if wl.prenorm_residual else x64
            check_route(wl, ref.cfg, ref.router_w, ref.router_b, xin, ih[t], wh[t],
                        where=f"noalloc {wl.name} call {call} t={t}")
    layer.close()


def test_route_noalloc_rejects_out_of_range(moe):
    wl = synth.WORKLOADS["tiny"]
    cfg = moe.make_config(wl.H, wl.E, wl.K, wl.I, wl.n_shared, wl.I_shared, wl.routed_scale)
    rw = torch.zeros((wl.E, wl.H), device="cuda")
    rb = torch.zeros(wl.E, device="cuda")
    x = torch.zeros((16, wl.H), device="cuda")
    idx = torch.zeros((16, wl.K), dtype=torch.int32, device="cuda")
    w = torch.zeros((16, wl.K), device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route_noalloc(cfg, rw, rb, x, moe.MOE_ROUTE_NOALLOC_MAX_TOKENS + 1, idx, w)
    assert e.value.status == moe.MOE_ERR_INVALID
    big = moe.make_config(wl.H, 2048, wl.K, wl.I, wl.n_shared, wl.I_shared, wl.routed_scale)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route_noalloc(big, rw, rb, x, 1, idx, w)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
