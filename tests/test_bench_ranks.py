"""bench.py's multi-rank plumbing (replicas: barrier + max over ranks), run as
world-size-2 gloo process groups on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world)  # rank 1 is the slower one
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)
    assert bench.packed_bytes(5120, 5120) == 5120 * 1280 + 5120 * 40 * 2
    assert bench.packed_bytes(5120, 27648, "base3") == 5120 * 5536 + 5120 * 216 * 2
    assert bench.step_bytes() == 64 * (2 * bench.packed_bytes(5120, 5120) + 2 * bench.packed_bytes(27648, 5120)
                                       + bench.packed_bytes(5120, 27648))
