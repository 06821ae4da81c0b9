"""Host logic of the multi-rank bench (one process per GPU, no collective on the data
path): two ranks over the gloo backend on CPU.  Checks the max-over-ranks reduction of
the timed totals, the barrier, and that the ranks' token streams are disjoint, so that
the whole-job value counts every rank's tokens once."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank's timed total; the job's time is the slowest rank's
        local_ms = 10.0 + 5.0 * rank
        job_ms = bench.reduce_max(local_ms, True)
        bench.barrier(True)
        streams = bench.rank_streams(rank, world, bench.N_X)
        q.put((rank, job_ms, streams))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_reduction_and_streams():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    # max over ranks, seen identically by every rank
    assert [o[1] for o in out] == [15.0, 15.0]
    # disjoint token streams per rank (weak scaling: each rank its own batches)
    s0, s1 = set(out[0][2]), set(out[1][2])
    assert len(s0) == len(s1) == len(out[0][2])
    assert not (s0 & s1)


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, False) == 3.5
    bench.barrier(False)
    assert bench.rank_streams(0, 1, 4) == [0, 1, 2, 3]
