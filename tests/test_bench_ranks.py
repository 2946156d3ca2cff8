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


def test_reference_arm_json_contract():
    """`bench.py --impl reference` (the CPU oracle on the host cores) prints one JSON line with
    the contract's keys, e2e without copies and a cpu_baseline describing the run."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "0", "--steps", "1",
                          "--warmup", "0"], cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["higher_is_better"] is False and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # the same config object our arm prints (built from the workload alone)
    args = bench.parse(["--config", "0"])
    assert line["config"] == json.loads(json.dumps(bench.bench_config(0, bench.workload_for(args), 1)))
    # what was timed is stated, and the timed region fits the steps it claims
    assert "whole" in line["sample"]
    assert line["wall_ms_timed_region"] >= line["value"] * line["steps"] * 0.99


def test_reference_arm_decoder_block_sample_is_bounded():
    """The default workload's reference arm times a bounded sample of the stated layer per step
    (seconds, not minutes) and reports any whole-layer estimate apart from `value`."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["config"]["workload"].startswith("llama3-8b-block")
    assert "q_proj" in line["config"]["stated_layer"] and "first 8 of 4096 rows" in line["sample"]
    assert line["value"] < 60_000
    assert line["extrapolated_stated_layer_ms"] > line["value"]
    assert "not measured" in line["extrapolation"]
