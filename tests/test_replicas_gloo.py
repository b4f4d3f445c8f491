"""The N > 1 bench path on CPU: two gloo ranks, each timing its own replica;
the job value uses the slowest rank and counts every rank's tokens."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    local_ms = [100.0, 250.0][rank]
    m = bench.max_over_ranks(local_ms, world)
    v = bench.replica_throughput(world, 4096, 10, m)
    dist.barrier()
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in out:
        assert m == 250.0
        assert v == pytest.approx(2 * 4096 * 10 / 0.25)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_throughput(1, 4096, 10, 500.0) == pytest.approx(81920.0)
