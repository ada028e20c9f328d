"""The benchmark drives one GPU.  A launch that asks for more (--gpus N > 1,
or WORLD_SIZE > 1 under torchrun) is refused before any device work: rank 0
prints one JSON line with the reason, the other ranks print nothing, and
every rank exits 0."""
import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, **env):
    e = dict(os.environ, **env)
    # no device for the child: a refusal must not need one
    e["CUDA_VISIBLE_DEVICES"] = ""
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=e,
                          capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("args,env", [(["--gpus", "2"], {}),
                                      (["--gpus", "8"], {"WORLD_SIZE": "8", "RANK": "0"})])
def test_multi_gpu_launch_is_refused_on_rank_0(args, env):
    r = _run(args, **env)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["n_gpus"] >= 2 and "single-GPU" in line["unavailable"]
    assert "value" not in line


def test_other_ranks_exit_quietly():
    r = _run(["--gpus", "2"], WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_job_throughput():
    assert bench.job_throughput(100, 2, 1000.0) == pytest.approx(200.0)
