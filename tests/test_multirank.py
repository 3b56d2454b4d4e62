"""The N>1 bench path (independent replicas, max-over-ranks timing) on CPU with gloo ranks."""
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import bench

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        r = bench.Ranks(dist, torch.device("cpu"))
        r.barrier()
        ms_local = 10.0 + 5.0 * rank          # the slowest rank defines the job time
        work_local = 1e12                     # every replica does the same work
        q.put((rank, r.max(ms_local), r.sum(work_local), r.rate(work_local, ms_local)))
        r.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_replica_aggregation_over_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = 10.0 + 5.0 * (world - 1)
    for rank, mx, sm, rate in out:
        assert mx == slowest
        assert sm == world * 1e12
        assert rate == pytest.approx(world * 1e12 / (slowest * 1e-3))


def test_single_process_has_no_collective():
    import bench

    r = bench.Ranks()
    assert r.max(3.0) == 3.0 and r.sum(2.0) == 2.0
    assert r.rate(1e12, 1.0) == pytest.approx(1e15)
