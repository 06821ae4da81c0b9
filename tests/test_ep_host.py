"""Expert parallelism, host side (no GPU): the ownership rule, the config checks,
and two gloo ranks on CPU whose partial outputs (computed by the oracle for the
experts each rank owns) are summed by the library's reduction and must equal
the oracle's whole layer.  The partition of the weighted sum over ranks is
what the pages' tiered residency relies on (reader.mx section 13)."""
import ctypes as C
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import int4_moe_expert_gb300 as m
    return m


def test_owned_ranges_partition_the_experts():
    from int4_moe_expert_gb300.expert_parallel import owned_range
    for E in (1, 16, 64, 256, 300):
        for W in range(1, min(E, 9) + 1):
            rs = [owned_range(E, W, r) for r in range(W)]
            assert rs[0][0] == 0 and rs[-1][1] == E
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))      # contiguous, disjoint
            sizes = [hi - lo for lo, hi in rs]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    for bad in ((16, 0, 0), (16, 17, 0), (16, 2, 2), (16, 2, -1)):
        with pytest.raises(ValueError):
            owned_range(*bad)


def test_ep_config_checked_before_any_device_work(moe):
    L = moe.lib()
    h = C.c_void_p(123)
    for size, rank in ((2, 2), (2, -1), (17, 0), (-1, 0)):
        cfg = moe.make_config(256, 16, 2, 128, 1, 128, 2.5, ep_size=size, ep_rank=rank)
        assert L.moe_init(C.byref(cfg), None, 1, C.byref(h)) == moe.MOE_ERR_INVALID
        assert "ep_size" in moe.moe_last_error()
        assert h.value is None


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, name, T, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import synth
    from int4_moe_expert_gb300.expert_parallel import owned_range, reduce_partials
    from parity_util import oracle_ep_partial
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.WORKLOADS[name]
        li = synth.layer_inputs(wl)
        x = synth.tokens(wl, T=T, stream=3)
        lo, hi = owned_range(wl.E, world, rank)
        part = np.stack([oracle_ep_partial(wl, li, x[t], lo, hi, rank == 0) for t in range(T)])
        y = torch.from_numpy(part.copy())
        reduce_partials(y)
        q.put((rank, part, y.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,world", [("tiny", 2), ("stack35b", 2), ("tiny", 3)])
def test_gloo_ranks_sum_to_the_whole_layer(name, world):
    """world ranks on CPU: every rank ends with the same y, equal (double
    rounding) to the oracle's layer; rank 0 alone carries the shared expert and
    the residual, and a rank's partial has only its own experts."""
    import multiprocessing as mp
    import oracle
    import synth
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from parity_util import oracle_layer
    oracle.build()
    T = 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, name, T, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted([q.get(timeout=300) for _ in range(world)], key=lambda o: o[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = synth.WORKLOADS[name]
    li = synth.layer_inputs(wl)
    x = synth.tokens(wl, T=T, stream=3)
    y_ref, idx, _, _ = oracle_layer(wl, li).forward(x)
    for _, _, y in out:
        assert np.array_equal(y, out[0][2])                      # one result on every rank
        np.testing.assert_allclose(y, y_ref, rtol=0, atol=1e-12 * np.abs(y_ref).max())
    # a rank whose experts none of the tokens selected holds exactly 0 (no shared, no x)
    from int4_moe_expert_gb300.expert_parallel import owned_range
    for r, part, _ in out[1:]:
        lo, hi = owned_range(wl.E, world, r)
        for t in range(T):
            if not any(lo <= e < hi for e in idx[t]):
                assert not part[t].any()
