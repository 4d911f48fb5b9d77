"""Host-side check of the streaming kernel's launch plans (no GPU needed).

Compiles tests/host/plan_check.cu -- which includes the kernel source and calls
its planner -- with nvcc for the host, then runs it over ~1.1M plans (hidden
8..16384 including ragged sizes, R 1..16, K 0..16, T 1..8192, every forced
cluster size, column-group count and slot size).  Any plan whose shared-memory layout, tile split,
thread coverage or transaction count is out of range fails the test."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_every_plan_is_in_range(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "plan_check"
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "tp_reduce_moe_gb300", "csrc"),
                    os.path.join(HERE, "host", "plan_check.cu"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "0 bad" in r.stdout
