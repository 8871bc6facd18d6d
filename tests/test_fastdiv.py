"""The kernels divide by plan-time divisors with a multiply-high and a shift (the round-up
method of Granlund and Montgomery, "Division by invariant integers using multiplication").
This compiles the library's own make_fastdiv (host code in csrc/internal.h) into a small
program that compares the result with hardware division over 11 million cases."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_include():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")


def test_fastdiv_matches_hardware_division(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(_cuda_include(), "cuda.h")):
        pytest.skip("needs g++ and the CUDA headers")
    exe = tmp_path / "fastdiv_check"
    subprocess.check_call([gxx, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "convolution_forward_implicit_gb300", "csrc"),
                           "-I", _cuda_include(), os.path.join(ROOT, "tests", "native", "fastdiv_check.cpp"),
                           "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert " 0 wrong" in out.stdout, out.stdout
