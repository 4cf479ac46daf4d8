"""Multi-rank host logic on CPU: two gloo ranks.

Each rank takes its contiguous token rows, aggregates them (with the oracle,
as the CPU stand-in for the per-GPU kernel: tokens are independent), and the
concatenation over ranks equals the unsharded result bit for bit; the
benchmark's timing reduction returns the max over ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from transformer_depth_wise_gb300.sharding import max_over_ranks, row_range, shard_rows


def test_row_range_partitions_exactly():
    for rows in (0, 1, 7, 64, 1001):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                a, b = row_range(rows, world, r)
                seen.extend(range(a, b))
                assert b - a in (rows // world, rows // world + 1)
            assert seen == list(range(rows))
    with pytest.raises(ValueError):
        row_range(10, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        g = torch.Generator().manual_seed(3)
        V = torch.randn(5, 2, 9, 16, generator=g, dtype=torch.float64)
        w = torch.randn(16, generator=g, dtype=torch.float64)
        mine = [shard_rows(v, world, rank).numpy() for v in V]
        h, _, _ = oracle.depth_aggregate(np.stack(mine), w.numpy(), None, 1e-8)
        parts = [None] * world
        dist.all_gather_object(parts, h)
        slowest = max_over_ranks(1.0 + rank)
        if rank == 0:
            full, _, _ = oracle.depth_aggregate(V.reshape(5, -1, 16).numpy(), w.numpy(), None, 1e-8)
            q.put((np.array_equal(np.concatenate(parts), full), slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_and_reduce_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    same, slowest = q.get(timeout=10)
    assert same and slowest == 2.0
