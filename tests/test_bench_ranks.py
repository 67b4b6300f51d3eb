"""bench.py's multi-replica logic on CPU: two gloo ranks (127.0.0.1), the max-over-ranks
reduction of the timings, and the reference arm running on rank 0 only."""
import argparse
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], "cpu")
        args = argparse.Namespace(workload="qwen3-14b-tiny", steps=1, warmup=0)
        ref = bench.run_reference(args, rank, world) if rank != 0 else "rank0-skipped"
        q.put((rank, got, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_only_rank0_runs_the_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, got, ref = q.get(timeout=120)
        res[rank] = (got, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        assert res[rank][0] == [2.0, 10.0, 3.5]
    assert res[1][1] is None   # a non-zero rank does no reference work and prints nothing


def test_reference_arm_line_carries_the_contract_keys():
    """The reference arm's JSON line (rank 0 of one): the metric and unit of our arm, the
    workload, a cpu_baseline describing the oracle run and an e2e object with no
    transfers."""
    import json

    args = argparse.Namespace(workload="qwen3-14b-tiny", steps=2, warmup=3)
    r = json.loads(json.dumps(bench.run_reference(args, 0, 1)))
    assert r["impl"] == "reference" and r["metric"] == bench.METRIC and r["unit"] == "us/step"
    assert r["higher_is_better"] is False and r["n_gpus"] == 1
    assert r["steps"] == 2 and r["warmup"] == 3 and r["config"] == bench.workload_config("qwen3-14b-tiny")
    assert r["config"]["workload"] == "qwen3-14b-tiny" and r["config"]["layers"] == 1
    assert r["value"] > 0 and r["ms_per_step"] == pytest.approx(r["value"] / 1e3, abs=1e-3)
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == r["value"] and cb["cores"] >= 1 and cb["sample"]
    assert r["e2e"] == {"value": r["value"], "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
