"""Per-device host state of the library (kd_host_state.h), checked on the CPU.

The library keeps kernel attributes, resident-cluster counts and SM counts per device
ordinal, set up on first use from whichever host thread gets there first.  This test
compiles a small C++ driver against that header with the host compiler and runs it:
16 threads over 8 device ordinals, a set-up that fails three times before it succeeds,
out-of-range ordinals, and a reset.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_teacher_kl_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "native", "host_state_check.cpp")


def test_per_device_state_from_many_threads(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "host_state_check")
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, SRC, "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
