"""The benchmark's multi-rank host logic on CPU with gloo, world size 2: the
slowest rank's time is taken (max over ranks), throughput is the units all
ranks processed over that time, and every rank gets its own batch of the
same shape (weak scaling, no data-path collective)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 1.0 + rank  # rank 1 is the slow one
        mx = bench.reduce_max(elapsed, torch, "cpu")
        wl = bench.rank_workload("gqa_video", rank, world)
        value = bench.aggregate(wl.tokens, world, mx, steps=10)
        q.put((rank, mx, value, wl.seed, wl.tokens, wl.algorithmic_bytes()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    (_, mx0, v0, s0, t0, b0), (_, mx1, v1, s1, t1, b1) = res
    assert mx0 == mx1 == 2.0
    assert v0 == v1 == pytest.approx(2 * 16384 * 10 / 2.0)
    assert s0 != s1 and t0 == t1 and b0 == b1


def test_single_process_reduce_is_identity():
    assert bench.reduce_max(3.5, torch, "cpu") == 3.5
    assert bench.aggregate(100, 1, 2.0, 4) == 200.0
