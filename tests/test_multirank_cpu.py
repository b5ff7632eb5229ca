"""The benchmark's multi-rank host logic on two CPU ranks (gloo).

On GPUs the benchmark runs one process per GPU under torchrun, each on its
own seeded batch (independent (sequence, head) work, weak scaling); the only
collectives are the timing barrier and the max-over-ranks reduction of the
step time. These tests run exactly those helpers with world size 2 on the
gloo backend, and the reference arm's rank discipline (rank 0 alone prints).
"""
import json
import os
import socket
import subprocess
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


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.rank_env()
        # a slow rank and a fast rank: the job time is the slow one's
        local_ms = 10.0 + 5.0 * r
        job_ms = bench.max_over_ranks(local_ms, w, torch.device("cpu"))
        dist.barrier()
        tokens = 4 * 4096
        value = bench.job_tokens_per_s(w, tokens, job_ms / 1e3)
        # each rank's batch is its own: the seeds and the drawn inputs differ
        from kda_gated_delta_chunkwise_gb300 import workloads as W
        x = W.batched(1, 8, 2, 16, 16, dtype="fp32", seed=bench.shard_seed(r))
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"env": [w, r, lr], "job_ms": job_ms, "value": value,
                       "q_sum": float(x.q.double().sum())}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["env"] == [2, r, r]
        assert d["job_ms"] == 15.0                    # max over ranks, seen by every rank
        assert d["value"] == pytest.approx(2 * 4 * 4096 / 0.015)
    assert res[0]["q_sum"] != res[1]["q_sum"]         # independent batches


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_tokens_per_s(1, 100, 0.5) == 200


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_json_line_follows_the_contract():
    """At N=1 the reference arm (the oracle on the host cores) prints one JSON
    line with the keys the benchmark contract names and the same metric and
    workload as the device arm."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    for key, val in bench.bench_config(1).items():  # the device arm's workload, plus the sample it times
        assert d["config"][key] == val, key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
