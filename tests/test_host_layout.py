"""Host-side invariants of the tensor-core offset-convolution backward
(window plan, accumulator-order layout of the grad_w_off partials), checked
by a small host program compiled from the kernel's own source over a sweep of
layer geometries.  Needs nvcc, no GPU."""
import os
import shutil
import subprocess

import pytest

from deformable_convolution_gb300 import _native as N

HERE = os.path.dirname(os.path.abspath(__file__))


def test_k4_plan_and_partials_layout(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "k4_layout_check")
    src = os.path.join(HERE, "host", "k4_layout_check.cu")
    subprocess.run([nvcc, *N.ARCH_FLAGS, "-O1", "-std=c++17", "-I", N.INCLUDE, src, "-o", exe],
                   check=True, capture_output=True, text=True, timeout=600)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert "0 failures" in r.stdout
