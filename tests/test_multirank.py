"""The multi-rank (torchrun) path of bench.py, on CPU with gloo, world size 2.

The forward has no exchange step, so ranks are independent replicas; the only
collective is the timing reduction: the job's time is the slowest rank's.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput(1e12, total, steps=2, world=world)
        out[rank] = (total, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
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
    assert res[0][0] == res[1][0] == 15.0          # the slowest rank's total
    # 2 ranks x 1e12 FLOPs per step, 7.5 ms per step
    assert res[0][1] == pytest.approx(2 * 1e12 / 7.5e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1e12, 10.0, steps=10, world=1) == pytest.approx(1000.0)
