"""bench.py's multi-process path on the CPU: two gloo ranks on 127.0.0.1 (the GPU run uses
NCCL with one rank per GPU; the replicas never exchange data, only the barrier and the
max-over-ranks time)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    ms = 10.0 + 5.0 * rank           # rank 1 is the slow replica
    worst = bench.max_over_ranks(ms, world)
    value = bench.job_value(8 * 1024, world, worst)
    out[rank] = (worst, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica_and_sum_the_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        worst, value = res[r]
        assert worst == 15.0                                  # max over ranks
        assert value == pytest.approx(8 * 1024 * 2 / 0.015)  # both ranks' tokens / slowest time


def test_single_process_path_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_value(100, 1, 1000.0) == pytest.approx(100.0)
