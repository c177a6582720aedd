"""Host logic of the multi-rank benchmark on two gloo ranks (CPU only).

Every output pixel is independent, so ranks shard by running their own
workload (weak scaling) with no collective on the data path; the only
exchange is the max over ranks of the measured time."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(0.5 + rank, world)           # rank 1 is the slower one
        rate = bench.whole_job_rate(100.0, world, t)
        results[rank] = (t, rate)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_rate():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        t, rate = results[r]
        assert t == 1.5                      # every rank sees the slowest time
        assert rate == pytest.approx(200.0 / 1.5)


def test_single_rank_is_identity():
    assert bench.reduce_max(0.25, 1) == 0.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def _run_reference(extra_env=None):
    env = dict(os.environ, **(extra_env or {}))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "2", "--warmup", "3", "--reference-step-seconds", "0.05"]
    return subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)


def test_reference_arm_prints_one_json_line():
    r = _run_reference()
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_reference({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
