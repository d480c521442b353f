"""The benchmark's host-side launch rules, on CPU: its own arm measures one
GPU and refuses a multi-rank launch before touching a GPU; its reference arm
(the oracle) runs on rank 0 alone and the other ranks exit 0 without work."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, **env):
    e = dict(os.environ, CUDA_VISIBLE_DEVICES="", **env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=e, cwd=ROOT,
                          capture_output=True, text=True, timeout=300)


def test_multi_rank_launch_is_refused():
    r = _bench(["--steps", "2", "--warmup", "3"], WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    assert r.returncode == 2
    assert "one GPU" in r.stderr and r.stdout == ""
    r1 = _bench(["--steps", "2", "--warmup", "3"], WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    assert r1.returncode == 2 and r1.stderr == "" and r1.stdout == ""


def test_more_than_one_gpu_flag_is_refused():
    r = _bench(["--gpus", "4", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 2 and "one GPU" in r.stderr


def test_reference_arm_skips_ranks_other_than_zero():
    r = _bench(["--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"],
               WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    r = _bench(["--impl", "reference", "--workload", "tiny_ref", "--steps", "2", "--warmup", "3",
                "--ref-budget", "3"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
