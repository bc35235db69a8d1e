"""The kernels' grid order (grid_pos / l2_group in kernels.cuh), checked as
host code: a bijection onto (tile, split, problem) for every group size, with
the plain order when one group holds every problem.  Needs nvcc, no GPU."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_grid_order_is_a_bijection():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = os.path.join(ROOT, "tests", "native", "grid_order_check.cu")
    inc = os.path.join(ROOT, "exact_attention_67_gb300", "csrc")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "grid_order_check")
        subprocess.run([nvcc, "-std=c++17", "-O1", "-I", inc, "-o", exe, src], check=True, capture_output=True)
        r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " 0 mismatches" in r.stdout
