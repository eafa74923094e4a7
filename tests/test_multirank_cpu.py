"""The benchmark's multi-process harness on CPU: two gloo ranks.

Rows are independent, so N GPUs run N replicas with no collective on the data
path; what has to work across ranks is the barrier, the max-over-ranks time
and the whole-job aggregate, which this test exercises with gloo.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), GBCE_DIST_BACKEND="gloo")
    import sys

    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 * (rank + 1), w, "cpu")
    value = bench.aggregate_gbs(w, 1_000_000_000, 4, slowest)
    out.put((rank, slowest, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_time_by_the_slowest_and_aggregate():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's 20 ms; 2 ranks x 4 steps x 1 GB in 20 ms
    assert [r[1] for r in results] == [20.0, 20.0]
    assert results[0][2] == pytest.approx(2 * 4 * 1.0 / 0.020)


def test_single_rank_needs_no_process_group():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.aggregate_gbs(1, 2_000_000_000, 10, 1000.0) == pytest.approx(20.0)
