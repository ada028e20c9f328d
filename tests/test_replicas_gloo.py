"""The multi-GPU path of the benchmark runs independent replicas (one per
GPU, no data-path collective).  Its only cross-rank steps are the barrier and
the max-over-ranks of the timings; checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r measured (100 + 10 r) ms device time and (150 - 20 r) ms end to end
    mine = [100.0 + 10 * rank, 150.0 - 20 * rank]
    dist.barrier()
    got = bench.max_over_ranks(mine, dist, device="cpu")
    q.put((rank, got, bench.job_throughput(16384, 5, world, got[0])))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tput in out:
        assert got == [110.0, 150.0]                      # max over both ranks, per entry
        assert tput == pytest.approx(2 * 16384 * 5 / 0.110)  # both ranks' tokens / slowest time


def test_single_process_is_identity():
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_throughput(100, 2, 1, 1000.0) == pytest.approx(200.0)
