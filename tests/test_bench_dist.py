"""The benchmark's multi-rank logic on CPU: two gloo ranks, slowest-rank time and
summed work (every rank runs its own copy of the workload; no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        bench.barrier(w)
        t, u = bench.aggregate(0.5 + rank, 32 * (rank + 1), w, device=None)
        q.put((r, w, t, u))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 1.5, 96), (1, 2, 1.5, 96)]


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(2.0, 7, 1) == (2.0, 7)
