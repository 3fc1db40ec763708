"""Replicas (the multi-GPU form of this layer: rows are independent, so each
GPU runs its own copy with no collective on the data path).  The bench's
cross-rank pieces run here on world size 2 with gloo on the CPU: the slowest
replica's time counts, throughput adds up over replicas, and each replica
draws its own layers and rows."""
from __future__ import annotations

import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q) -> None:
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t = bench.reduce_max(1.5 + rank)  # rank 1 is the slower replica
        q.put((rank, t, bench.rows_per_second(world, 10, 3, t), bench.replica_seed(7, rank)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_throughput_and_seeds():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2.5 for r in res)            # the max over ranks
    assert all(r[2] == pytest.approx(2 * 10 * 3 / 2.5) for r in res)
    assert res[0][3] != res[1][3]                   # independent work per replica
    assert all(p.exitcode == 0 for p in procs)


def test_single_process_needs_no_group():
    import bench
    assert bench.reduce_max(3.25) == 3.25
    assert bench.rows_per_second(1, 4, 2, 2.0) == 4.0
