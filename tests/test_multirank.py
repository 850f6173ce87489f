"""Multi-rank host logic of the benchmark, as world-size-2 gloo ranks on CPU.

The verify step shards by sequence with no data-path exchange; across ranks
only the timing is reduced: the step time is the max over ranks and the
positions are summed.  This runs the same helpers bench.py uses.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    bench.init_dist(ws, "gloo")
    try:
        step_ms = [3.0, 5.0][r]              # rank 1 is the slow one
        positions = [40, 40][r]
        t = bench.max_over_ranks(step_ms, ws)
        n = bench.sum_over_ranks(positions, ws)
        bench.barrier(ws)
        q.put((r, ws, t, n))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_reduce_time_and_positions():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for r, ws, t, n in res:
        assert ws == 2
        assert t == 5.0                     # max over ranks
        assert n == 80                      # whole-job positions
    # the whole-job rate counts every rank's work against the slowest rank
    assert 80 / (5.0e-3) == pytest.approx(16000.0)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.sum_over_ranks(7, 1) == 7.0
    assert bench.dist_env()[0] == int(os.environ.get("WORLD_SIZE", "1"))
