"""The multi-process bench logic on CPU: two gloo ranks, max-over-ranks timing
and the weak-scaling aggregate (rows are independent: no data collective)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        got = bench.reduce_max(local_ms, torch.device("cpu"))
        rows = bench.weak_scaling_rows_per_s(world, 64, 20, got)
        q.put((rank, got, rows))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_scale_weakly():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, got, rows in res:
        assert got == pytest.approx(15.0)
        assert rows == pytest.approx(2 * 64 * 20 / 15e-3)


def test_single_process_is_identity():
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    assert bench.weak_scaling_rows_per_s(1, 64, 10, 100.0) == pytest.approx(6400.0)
