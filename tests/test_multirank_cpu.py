"""World-size-2 gloo test of bench.py's multi-rank host logic on CPU: every
rank runs an independent replica, the job time is the slowest rank's, and the
job throughput counts every replica's work."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    out[rank] = bench.max_over_ranks(ms, world, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == pytest.approx(15.0) and out[1] == pytest.approx(15.0)


def test_job_throughput_counts_every_replica():
    flops = 2.2e13
    assert bench.job_throughput(flops, 1, 14.0) == pytest.approx(flops / 14e-3 / 1e12)
    assert bench.job_throughput(flops, 4, 14.0) == pytest.approx(4 * flops / 14e-3 / 1e12)
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
