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


def test_shard_range_covers_the_batch():
    import bench
    for n in (1, 7, 8, 32, 257):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_range(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [e - s for s, e in spans]
            assert max(sizes) - min(sizes) <= 1


def _accept_worker(rank, world, port, out, n, k, V):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from oracle import accept as A
    from synthetic import make_accept_inputs
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        start, stop = bench.shard_range(n, world, rank)
        p, q, x, u = make_accept_inputs(stop - start, k, V, seed=2, first=start)
        mine = [(start + b,) + tuple(int(v) for v in A.accept_sampling_chain(p[b], q[b], x[b], u[b]))
                for b in range(stop - start)]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        out[rank] = [r for part in gathered for r in part]
    finally:
        dist.destroy_process_group()


def test_sharded_acceptance_equals_the_unsplit_batch():
    """The batched workloads split one global batch over the ranks by
    shard_range; every rank draws only its own sequences (streams keyed by the
    global index) and runs the oracle's rejection sampling on them.  Gathered,
    the per-sequence decisions equal those of the undivided batch."""
    from oracle import accept as A
    from synthetic import make_accept_inputs
    n, k, V = 7, 3, 64
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_accept_worker, args=(r, 2, port, out, n, k, V)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    p, q, x, u = make_accept_inputs(n, k, V, seed=2)
    want = [(b,) + tuple(int(v) for v in A.accept_sampling_chain(p[b], q[b], x[b], u[b])) for b in range(n)]
    assert res[0] == res[1] == want
