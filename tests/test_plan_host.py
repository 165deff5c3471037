"""Host-side launch planning (csrc/bl_plan.h), compiled with g++ and checked
over a grid of shapes (no GPU needed)."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plan_invariants(tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("g++ unavailable")
    exe = tmp_path / "plan_check"
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-I",
                           os.path.join(ROOT, "w1_a8_bitlinear_02_b300", "csrc"),
                           os.path.join(ROOT, "tests", "host", "plan_check.cpp"), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok:")
    # the ~2B and 100B decode shapes at M = 1 run on the GEMV path
    for line in ("M=1 K=2560 path=gemv", "M=1 K=6912 path=gemv", "M=1 K=28672 path=gemv"):
        assert line in out.stdout
