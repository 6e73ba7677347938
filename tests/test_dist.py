"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank
runs its own replica, the job time is the slowest rank's, and the job value is
the aggregate over ranks.  No GPU and no data-path collective are involved."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    assert bench.dist_env() == (world, rank, rank)
    ms = [1200.0, 1500.0][rank]
    job_ms = bench.max_over_ranks(ms, torch.device("cpu"))
    value = bench.job_throughput(1e15, world, job_ms)
    out[rank] = (job_ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        job_ms, value = res[r]
        assert job_ms == 1500.0
        assert value == pytest.approx(1e15 * 2 / 1.5 / 1e12)


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.0, torch.device("cpu")) == 3.0
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)
