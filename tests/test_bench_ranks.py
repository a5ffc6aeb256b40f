"""bench.py's multi-rank logic on CPU: world_size 2 over gloo.

Ranks are independent replicas (weak scaling, no data-path collective); the
only exchange is the max over ranks of the timed region, which the job's
throughput divides into. Run here as two gloo processes on 127.0.0.1.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        m = bench.max_over_ranks(times[rank], dist)
        out[rank] = m
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.25, 0.4), (1.5, 0.75)])
def test_max_over_ranks_gloo_world2(times):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == max(times)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.125) == 0.125


def test_weak_scaling_throughput():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 256 sequences x 10 steps in the slowest rank's 0.5 s
    assert bench.job_throughput(2, 256, 10, 0.5) == 2 * 256 * 10 / 0.5
    assert bench.job_throughput(1, 256, 10, 0.5) * 2 == bench.job_throughput(2, 256, 10, 0.5)
