"""CPU check of the library's own rotary sin/cos (rope_math.cuh).

The norm/RoPE kernel forms each angle pos * inv_freq and reduces it by
quarter turns in float64, then evaluates sin and cos in float-float
arithmetic on the float32 pipe (a 51-knot table and the addition theorems).
Compiled here as host code (no multiply-add contraction, like the device
build's separately rounded operations) and compared with the C library's
long-double sin/cos: the reduced-angle evaluation over 2M angles in
[-pi/4, pi/4] (every quadrant, knot edges included) must be within 1e-13
absolute, as the rotation's cancellation analysis needs; the whole path on
RoPE angles (theta 1e6, positions up to 65535) within 1e-11, the float64
rounding of pos * inv_freq itself being the larger part.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "rope_math_check.cu")


def test_rotary_sincos_against_long_double(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "rope_math_check"
    subprocess.run([nvcc, "-O2", "-std=c++17", "-Xcompiler", "-ffp-contract=off", "-o", str(exe),
                    SRC], check=True,
                   stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    out = subprocess.run([str(exe), "2000000"], check=True, stdout=subprocess.PIPE).stdout.decode()
    es, ec, fs, fc = (float(x) for x in out.split()[:4])
    assert es <= 1e-13 and ec <= 1e-13, out
    assert fs <= 1e-11 and fc <= 1e-11, out
