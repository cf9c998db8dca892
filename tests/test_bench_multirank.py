"""The bench's N>1 host path on CPU: two gloo ranks (127.0.0.1) reduce their
per-rank times to the slowest one and form the whole-job throughput from it,
as the GPU launch does over NCCL (one independent replica per GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_s = [0.25, 0.5][rank]                    # rank 1 is the slowest
        slowest = bench.reduce_max(local_s, dist, "cpu")
        out[rank] = (slowest, bench.job_rate(world, 10, slowest))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1] == pytest.approx((0.5, 40.0))


def test_job_rate_single_rank():
    import bench
    assert bench.job_rate(1, 5 * 50, 0.5) == 500.0
