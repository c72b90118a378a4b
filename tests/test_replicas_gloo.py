"""The N > 1 path of bench.py on CPU: independent replicas, slowest rank's time.

Two processes join a gloo group on 127.0.0.1 and reduce their own timings
through bench.job_rate, as the GPU ranks do over NCCL: both must see the
maximum and the same whole-job rate (all ranks' rounds over that time).
"""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
    ms, value = bench.job_rate(local_ms, steps=20, world=world, dist=dist)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_job_rate_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 150.0
        assert value == pytest.approx(2 * 20 / 0.150)


def test_job_rate_single_rank_is_local():
    import bench
    ms, value = bench.job_rate(40.0, steps=10, world=1)
    assert ms == 40.0 and value == pytest.approx(250.0)
