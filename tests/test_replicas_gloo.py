"""The N > 1 bench path on CPU: replicas time their own regions, the job takes
the max over ranks, and the whole-job throughput counts every rank's tokens
(two gloo ranks on 127.0.0.1, no GPU)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (10 + r) ms for the timed region, (12 - r) ms end to end
        region, e2e = bench.job_times([10.0 + rank, 12.0 - rank], world, "cpu")
        out[rank] = (region, e2e, bench.job_throughput(64 * 8 * world, region))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_all_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        region, e2e, thr = res[r]
        assert region == pytest.approx(11.0)      # max of 10 and 11
        assert e2e == pytest.approx(12.0)         # max of 12 and 11
        assert thr == pytest.approx(64 * 8 * 2 / 0.011)
