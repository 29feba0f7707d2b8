"""bench.py's multi-GPU bookkeeping with two gloo ranks on the CPU.

Under torchrun every GPU runs an independent replica of the step (the method
itself is simulated inside each GPU), so the only cross-rank traffic is the
barrier and the timing aggregation: the job's time is the slowest rank's and
its work is the sum over ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    step_ms = [2.0, 3.5][rank]          # the slower rank decides the job's time
    work = [10.0, 30.0][rank]
    slowest = bench.max_over_ranks(dist, step_ms)
    total = bench.sum_over_ranks(dist, work)
    bench.barrier(dist)
    dist.destroy_process_group()
    out.put((rank, slowest, total))


@pytest.mark.timeout(120)
def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert results == [(0, 3.5, 40.0), (1, 3.5, 40.0)]


def test_single_process_needs_no_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 1.25) == 1.25
    assert bench.sum_over_ranks(None, 2.5) == 2.5
