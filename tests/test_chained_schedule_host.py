"""Host check of the chained k-split's schedule: the same SkPlan code the
GEMM kernel runs, compiled for the host with nvcc, walked for every worker of
many (tiles, k-slices, workers) cases.  Every (tile, slice) must run exactly
once; a split tile's chain must be continued by the next worker exactly where
the previous one's head stopped; no tail may come before the head it
continues is done (in slice counts: no wait when the workers run at one
speed)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "verifiable_repops_gemm_gb300", "csrc")


def test_chained_schedule_invariants(tmp_path):
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "chained_schedule_check")
    cmd = [nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
           os.path.join(HERE, "host", "chained_schedule_check.cu"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok "), r.stdout
    assert int(r.stdout.split()[1]) > 20000
