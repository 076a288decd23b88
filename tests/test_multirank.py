"""Multi-process timing aggregation of bench.py, on CPU with the gloo backend
(world size 2): the job's time is the slowest rank's, and throughput counts
every rank's independent batch (weak scaling, no collective on the data)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        thr = bench.job_throughput(1000, world, slowest)
        out[rank] = (slowest, thr)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_units():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    slowest, thr = res[0]
    assert slowest == 20.0
    assert thr == pytest.approx(2 * 1000 / 0.020)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.job_throughput(100, 1, 10.0) == pytest.approx(10000.0)
