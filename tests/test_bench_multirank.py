"""bench.py across ranks (replicas): the whole-job value is the units summed
over ranks divided by the slowest rank's time.  Two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        units = 1000.0 * (rank + 1)   # ranks did different amounts of work
        secs = 0.5 + 0.25 * rank      # and the slowest took 0.75 s
        ws, r, _ = bench.dist_info()
        value, secs_max, units_all = bench.aggregate(units, secs, ws, bench.torch_reduce_fn("cpu"))
        q.put((r, value, secs_max, units_all))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_sum_over_max():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for r, value, secs_max, units_all in got:
        assert units_all == pytest.approx(3000.0)
        assert secs_max == pytest.approx(0.75)
        assert value == pytest.approx(4000.0)


def test_single_rank_aggregate_is_plain_rate():
    import bench

    assert bench.aggregate(500.0, 0.25, 1) == (2000.0, 0.25, 500.0)
