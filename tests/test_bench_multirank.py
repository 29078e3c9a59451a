"""bench.py's multi-rank plumbing on CPU: two gloo ranks, barrier, the
max-over-ranks timing and the summed whole-job units (replicas, no collective
on the data path)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.barrier(w)
    t = bench.max_over_ranks(1.0 + rank, w)       # the slowest rank sets the time
    units = bench.sum_over_ranks(100.0 * (rank + 1), w)  # every replica's tokens count
    q.put((rank, t, units))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert all(p.exitcode == 0 for p in procs)
    assert [x[1] for x in res] == [2.0, 2.0]
    assert [x[2] for x in res] == [300.0, 300.0]


def test_single_rank_helpers_are_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    bench.barrier(1)
