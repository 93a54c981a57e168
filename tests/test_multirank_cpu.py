"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks, each with
its own elapsed time; both must see the slowest rank's time, and the job
throughput counts every rank's steps over that time (replicas, weak scaling)."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.rank_env()
    mine = 10.0 + 5.0 * rank          # rank 1 is the slow one
    slowest = bench.max_over_ranks(mine, w)
    gbs = bench.job_throughput(bench.DECODE_BYTES, 100, w, slowest)
    q.put((r, lr, w, slowest, gbs))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    expect = bench.DECODE_BYTES * 100 * 2 / (15.0 / 1e3) / 1e9
    for rank, (r, lr, w, slowest, gbs) in enumerate(res):
        assert (r, lr, w) == (rank, rank, 2)
        assert slowest == 15.0
        assert abs(gbs - expect) < 1e-9 * expect


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1e9, 10, 1, 1000.0) == 10.0
