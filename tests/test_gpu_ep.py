"""Expert parallelism on the GPU (one device): W handles, one per rank, each
holding only its own experts (the others NULL) and run in turn on the same
tokens.  Every rank must make the same selection as the oracle, each rank's
partial must equal the oracle's partial for the experts it owns (plus the
shared expert and the residual on rank 0), and the partials summed in rank
order must equal the oracle's layer.  The all-reduce between GPUs itself is
covered on CPU (test_ep_host.py) and is not measured on hardware."""
import numpy as np
import pytest

import oracle
import synth
from parity_util import (REL_TOL, check_route, check_token, gpu_config, oracle_ep_partial,
                         oracle_layer)

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


def _cfg_kwargs(wl):
    return dict(H=wl.H, E=wl.E, K=wl.K, I=wl.I, n_shared=wl.n_shared, I_shared=wl.I_shared,
                routed_scale=wl.routed_scale, norm_topk=wl.norm_topk,
                prenorm_residual=wl.prenorm_residual, rms_eps=wl.rms_eps, n_group=wl.n_group,
                topk_group=wl.topk_group, score_func=wl.score_func,
                expert_format=wl.expert_format, shared_format=wl.shared_format)


@pytest.mark.parametrize("name,T,W", [
    ("tiny", 1, 2), ("tiny", 37, 3), ("stack35b", 1, 2), ("stack35b", 8, 4),
    ("olmoe_int8", 1, 2), ("group8", 5, 2), ("glm_decode", 1, 2), ("glm_batched", 300, 2),
])
def test_expert_parallel_partials(moe, name, T, W):
    from int4_moe_expert_gb300.expert_parallel import ExpertParallelLayer, owned_range
    wl = synth.WORKLOADS[name]
    li = synth.layer_inputs(wl)
    assert gpu_config(moe, wl).ep_size == 1     # the plain config is unchanged
    x = synth.tokens(wl, T=T, stream=21)
    xd = torch.from_numpy(x).cuda()
    ranks = [ExpertParallelLayer(_cfg_kwargs(wl), li.router_w, li.router_b, li.slabs, li.scales,
                                 li.sh_slab, li.sh_scale, ep_size=W, ep_rank=r, max_tokens=T)
             for r in range(W)]
    try:
        outs = []
        for rk in ranks:
            assert not moe.moe_uses_streaming_decode(rk.handle)
            outs.append(rk.layer.forward_debug(xd))
            assert moe.moe_device_error(rk.handle) == 0
        torch.cuda.synchronize()
        for y_r, idx_r, w_r in outs[1:]:            # one selection on every rank
            assert torch.equal(idx_r, outs[0][1]) and torch.equal(w_r, outs[0][2])
        parts = np.stack([o[0].cpu().numpy() for o in outs]).astype(np.float64)   # [W, T, H]
        idx, w = outs[0][1].cpu().numpy(), outs[0][2].cpu().numpy()
        total = torch.stack([o[0] for o in outs]).sum(0).cpu().numpy()           # rank order
        ref = oracle_layer(wl, li)
        cfg_o = ref.cfg
        for t in range(T):
            check_token(wl, ref, x[t], total[t], idx[t], w[t], where=f"{name} ep{W} sum t={t}")
        # per-rank partials on a few tokens, against the oracle's partial of the same rank
        for t in range(min(T, 6)):
            x64 = x[t].astype(np.float64)
            xin = oracle.rmsnorm(x64, wl.rms_eps) if wl.prenorm_residual else x64
            forced, _ = check_route(wl, cfg_o, li.router_w, li.router_b, xin, idx[t], w[t], f"{name} t={t}")
            y_full = ref.token(x64, forced_idx=forced)[0]
            den = max(np.abs(y_full).max(), 1e-30)
            for r in range(W):
                lo, hi = owned_range(wl.E, W, r)
                p_ref = oracle_ep_partial(wl, li, x[t], lo, hi, r == 0, idx=forced)
                e = float(np.abs(parts[r, t] - p_ref).max() / den)
                assert e <= REL_TOL, (name, W, r, t, e)
                if r > 0 and not any(lo <= i < hi for i in idx[t]):
                    assert not parts[r, t].any()    # neither shared expert nor residual off rank 0
    finally:
        for rk in ranks:
            rk.close()
