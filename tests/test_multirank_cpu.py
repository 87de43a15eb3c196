"""The bench's multi-rank path on CPU: two gloo ranks, no GPU.

Rows are independent, so N GPUs run N replicas with no collective on the data
path; the only cross-rank steps are the barrier around the timed region and
the max over ranks of the elapsed time. Both are exercised here with
world_size 2 over gloo on 127.0.0.1.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(0.5 + rank, w)   # rank 1 is the slow one
    q.put((rank, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 1.5), (1, 1.5)]


def test_single_rank_needs_no_process_group(monkeypatch):
    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    import bench
    assert bench.dist_setup(1) == (0, 1, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def _value_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(world)
    # Each rank ran 100 steps of 32 rows in its own time; the job's value
    # counts every rank's rows over the slowest rank's time.
    secs = bench.max_over_ranks(0.004 * (1 + r), w)
    q.put((r, bench.job_value(w, 32, 100, secs)))
    dist.destroy_process_group()


def test_whole_job_value_counts_every_rank_over_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_value_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    # 2 ranks x 32 rows x 100 steps over rank 1's 8 ms.
    assert got == [(0, pytest.approx(800000.0)), (1, pytest.approx(800000.0))]
