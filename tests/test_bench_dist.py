"""The benchmark's multi-rank logic on CPU: world size 2 over gloo, no GPU.

Each rank reports its own time; the job keeps the maximum (the slowest rank bounds the
whole job) and the weak-scaling value counts the work of all ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        times = bench.reduce_max([1.0 + rank, 10.0 - rank], w)
        q.put((r, w, local, times))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [r[:3] for r in results] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, times in results:
        assert times == [2.0, 10.0]


def test_single_rank_reduce_is_identity():
    import bench

    assert bench.reduce_max([3.0, 4.0], 1) == [3.0, 4.0]
    bench.barrier(1)
