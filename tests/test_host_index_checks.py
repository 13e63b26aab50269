"""The GEMMs' index arithmetic checked on the CPU (no GPU): nvcc compiles
tests/host_index_checks.cu, which calls the library's own __host__
__device__ helpers (pair-CTA tile order, stream-K ranges, TMEM accumulator
strides), and the binary runs on the host."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def test_host_index_checks(tmp_path):
    if not (os.path.exists(NVCC) or shutil.which("nvcc")):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "host_index_checks")
    src = os.path.join(ROOT, "tests", "host_index_checks.cu")
    cc = subprocess.run([NVCC, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", src, "-o", exe],
                        capture_output=True, text=True, timeout=300)
    assert cc.returncode == 0, cc.stdout + cc.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "host index checks: 0 failures" in r.stdout
