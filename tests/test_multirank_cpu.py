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


def _slice_worker(rank, world, port, out):
    # each rank holds one slice of the vocabulary; the partials of its slice
    # (the oracle's, on CPU) go through the library's gather helper, and the
    # merged result must be the full-row log-probs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import sys

    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist

    import cross_entropy_gb300 as gbce
    import oracle
    import workloads

    dist.init_process_group("gloo", rank=rank, world_size=world)
    V, T = 101, 0.8
    w = workloads.peaked_rows_tiny(V, [0.0, 17.0, 30.0, 50.0, 5.0], seed=9)
    x = w.logits.numpy()
    idx = np.stack([w.labels.numpy(), (w.labels.numpy() * 7 + 3) % V], axis=1)
    offsets = [0, 37, V] if world == 2 else [0, V]
    a, b = offsets[rank], offsets[rank + 1]
    m, s, xt = oracle.vocab_slice_partials(x[:, a:b], idx, a, T)
    mine = torch.from_numpy(np.concatenate([m[:, None], s[:, None], xt], axis=1))
    everyone = gbce.gather_slice_partials(mine)
    parts = [(p[:, 0].numpy(), p[:, 1].numpy(), p[:, 2:].numpy()) for p in everyone]
    got, _ = oracle.vocab_slice_combine(parts, offsets, idx, T)
    want, _ = oracle.selective_logsoftmax(x, idx, T)
    out.put((rank, tuple(everyone.shape), float(np.max(np.abs(got - want) / np.abs(want)))))
    dist.destroy_process_group()


def test_vocab_slices_gathered_across_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_slice_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, shape, err in results:
        assert shape == (2, 5, 4)      # [slices, rows, 2 + K], in rank order
        assert err <= 1e-13
