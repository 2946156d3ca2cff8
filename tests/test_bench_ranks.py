"""Host logic of bench.py's multi-rank path, on CPU with two gloo ranks.

Every rank runs its own replica of the layer pass (no data-path collective); the only
exchange is the max over ranks of the step time, and rank 0 alone prints. The reference
arm runs on rank 0 only: the other ranks return without work.
"""
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


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_info() == (ws, rank, rank)
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, ws, "cpu")   # rank 1 is the slow one
        out.put((rank, ms, bench.replica_value(ms, ws)))
        if rank != 0:
            # the reference arm: rank != 0 returns at once, without building anything
            assert bench.run_reference(bench.parse(["--impl", "reference"]), ws, rank) is None
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_and_report_per_replica():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 15.0, 7.5), (1, 15.0, 7.5)]


def test_single_rank_is_untouched():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.replica_value(3.25, 1) == 3.25
