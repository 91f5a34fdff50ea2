"""bench.py's multi-rank logic on CPU: two gloo ranks, each an independent
replica, combine to all ranks' tokens over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r takes (r + 1) x 10 ms per step over 4 steps of 1000 tokens
        times = [10.0 * (rank + 1)] * 4
        value, ms = bench.aggregate(1000, times, world, torch.device("cpu"))
        mx = bench.reduce_max(float(rank), world, torch.device("cpu"))
        bench.barrier(world)
        out[rank] = (value, ms, mx)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_over_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        for p in procs:
            if p.is_alive():
                p.kill()
                pytest.fail("gloo rank did not finish")
            assert p.exitcode == 0
        res = dict(out)
    # slowest rank: 4 x 20 ms = 80 ms; all ranks' tokens: 2 x 4 x 1000
    for r in range(world):
        value, ms, mx = res[r]
        assert ms == pytest.approx(20.0)
        assert value == pytest.approx(8000 / 0.080)
        assert mx == 1.0


def test_single_rank_aggregate():
    value, ms = bench.aggregate(500, [2.0, 4.0], 1, torch.device("cpu"))
    assert ms == pytest.approx(3.0)
    assert value == pytest.approx(1000 / 0.006)
