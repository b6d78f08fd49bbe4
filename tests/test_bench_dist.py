"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, no GPU.

Replicas only: every rank runs a full batch, the job's time is the slowest
rank's, and its throughput counts every rank's clips.  The reference arm does
its work on rank 0 alone.
"""
import json
import os
import pathlib
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = pathlib.Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(values[rank], world, "cpu")
        thr = bench.job_throughput(world, 256, 10, got)
        pathlib.Path(out_dir, f"r{rank}.json").write_text(json.dumps({"max": got, "thr": thr}))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    values = [2.5, 7.25]  # milliseconds: rank 1 is the slow one
    mp.start_processes(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.loads((tmp_path / f"r{r}.json").read_text()) for r in range(2)]
    assert res[0]["max"] == res[1]["max"] == 7.25
    # 2 ranks x 256 clips x 10 steps in 7.25 ms
    assert res[0]["thr"] == pytest.approx(2 * 256 * 10 / 7.25e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(1, 8, 4, 2.0) == pytest.approx(8 * 4 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_line(oracle_mod):
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--reference-clips", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "clips/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
