"""The multi-rank logic of bench.py on CPU: two gloo ranks.

Ranks are replicas (weak scaling): the job's time is the slowest rank's and
its throughput counts every rank's units.  No GPU, no data-path collective.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms for the step and 10 - r ms end to end
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == [2.0, 10.0] and out[1] == [2.0, 10.0]


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.5, 1]) == [3.5, 1.0]


def test_job_throughput_counts_every_rank():
    # 2 ranks x 1000 tokens in 2 ms -> 1e6 tokens/s for the job
    assert bench.job_throughput(2, 1000, 2.0) == pytest.approx(1e6)
    assert bench.job_throughput(1, 1000, 2.0) == pytest.approx(5e5)
