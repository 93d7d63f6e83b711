"""The bench's multi-rank path on CPU: two gloo ranks, barrier and max-over-ranks
timing, and the whole-job throughput computed from the slowest rank."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(backend="gloo")
    d.barrier()
    ms = d.max(1.0 + rank)  # rank 1 is the slow one
    q.put((rank, ms, bench.whole_job_gbps(1_000_000, d.world, ms)))
    d.close()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, ms, gbps in res:
        assert ms == 2.0
        assert gbps == pytest.approx(1_000_000 * 2 / 2e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(backend="gloo")
    assert d.world == int(os.environ.get("WORLD_SIZE", "1")) == 1
    assert d.max(3.5) == 3.5
    assert bench.whole_job_gbps(8192, 1, 1.0) == pytest.approx(8192 / 1e-3 / 1e9)
