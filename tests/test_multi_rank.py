"""Replicas across ranks on CPU (gloo, world size 2), launched the way the bench is launched for
several GPUs: the job's step time is the slowest rank's, the throughput counts every rank's
tokens, every rank draws its own batch, and the reference arm runs on rank 0 only."""
import json
import os
import re
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env():
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    return env


def test_two_gloo_ranks_take_the_slowest_step_and_count_all_tokens():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "tests", "multi_rank_worker.py")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=240, env=_env(), cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(m) for m in re.findall(r"\{[^{}]*\}", r.stdout)]  # the ranks share one stdout
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["slowest_ms"] == 15.0  # max over ranks
        assert abs(l["tokens_per_s"] - 2 * 4 * 2 / 0.015) < 1e-6
        assert l["distinct_tokens"]


def test_reference_arm_runs_on_rank_zero_only():
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1", "--layers", "1",
            "--steps", "1", "--warmup", "0"]
    env = _env()
    env.update({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    r1 = subprocess.run(args, capture_output=True, text=True, timeout=240, env=env, cwd=ROOT)
    assert r1.returncode == 0 and r1.stdout.strip() == "", r1.stderr[-2000:]
    env.update({"RANK": "0", "LOCAL_RANK": "0"})
    r0 = subprocess.run(args, capture_output=True, text=True, timeout=240, env=env, cwd=ROOT)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
