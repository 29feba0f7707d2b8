"""bench.py's host-side contract, on the CPU: one process on one GPU.

The library simulates every tensor-parallel rank on one GPU and its GEMMs
multicast operand tiles within a thread-block cluster of that GPU, so the
benchmark runs as a single process: asked for more GPUs, or started as one of
several torchrun ranks, it refuses with a clear message and a non-zero exit,
before it touches a GPU.  The CPU reference arm runs on rank 0 alone.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, env=None, timeout=120):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=e, timeout=timeout, cwd=ROOT)


def test_more_than_one_gpu_is_refused():
    r = _bench(["--gpus", "2", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 2
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["value"] is None and "single-GPU" in line["error"]


def test_torchrun_world_of_two_is_refused():
    r = _bench(["--steps", "3"], env={"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 2
    assert r.stdout.strip() == ""          # only rank 0 prints the line
    assert "WORLD_SIZE=2" in r.stderr


def test_reference_arm_other_ranks_exit_without_work():
    r = _bench(["--impl", "reference", "--steps", "3"], env={"WORLD_SIZE": "2", "RANK": "1"})
    assert r.returncode == 0
    assert r.stdout.strip() == ""
