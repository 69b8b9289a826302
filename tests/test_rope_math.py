"""CPU check of the decode library's own sin/cos (rope_math.cuh).

The norm/RoPE kernel evaluates sin and cos of the token's reduced angles with
its own Taylor-series routine (float64 leading terms, float32 tails) instead
of float64 sincos.  Compiled here as host code and compared with the C
library's long-double sin/cos over 2M angles in [-pi, pi] plus quarter-turn
boundaries: the rotation's cancellation analysis needs ~1e-13 absolute.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "rope_math_check.cu")


def test_sincos_reduced_against_long_double(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "rope_math_check"
    subprocess.run([nvcc, "-O2", "-std=c++17", "-o", str(exe), SRC], check=True,
                   stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    out = subprocess.run([str(exe), "2000000"], check=True, stdout=subprocess.PIPE).stdout.decode()
    es, ec = (float(x) for x in out.split()[:2])
    assert es <= 1e-13 and ec <= 1e-13, out
