"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own elapsed time,
agree on the slowest rank's time and on the whole-job rate (replicas, weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [0.5, 2.0][rank]
        slow = bench.max_over_ranks(mine, world)
        rate = bench.job_rate(10, world, slow)
        dist.barrier()
        out[rank] = (slow, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_rate():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 10.0)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_rate(30, 1, 0.5) == 60.0
