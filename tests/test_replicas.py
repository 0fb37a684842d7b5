"""The multi-GPU path is replicas only (no sharding, no collective on the data
path): bench.py under torchrun runs one independent step per rank, takes the
slowest rank's time and reports the whole job's tokens.  This checks that host
logic with two gloo ranks on the CPU."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(0.010 + 0.005 * rank, dist, "cpu")  # rank 1 is the slower replica
    out[rank] = (t, bench.job_throughput(8192, world, t))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_tokens():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == pytest.approx(0.015) and res[1][0] == pytest.approx(0.015)
    assert res[0][1] == pytest.approx(2 * 8192 / 0.015)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(0.02, None, "cpu") == 0.02
    assert bench.job_throughput(100, 1, 0.5) == 200
