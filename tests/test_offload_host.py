"""The offloaded step's host pipeline (zero_offload.cpp) on the CPU alone: a C++ driver
compiled against the library's host source checks the overlapped update against the plain
one bit for bit, the order and coverage of the ranges it hands back for the copy to the
device, and a clean stop when a wait for the gradient gives up."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "zero_sharded_mixed_03_gb300", "csrc")
sys.path.insert(0, ROOT)


def test_overlapped_host_update_matches_and_hands_back_every_range(tmp_path):
    from zero_sharded_mixed_03_gb300 import _build
    # the library's own host flags for this file (given to nvcc as -Xcompiler pairs)
    flags = [f for f in _build.EXTRA["zero_offload.cpp"] if f != "-Xcompiler"]
    exe = str(tmp_path / "offload_host_check")
    cmd = ["g++", "-O3", "-std=c++17", "-pthread", *flags, "-I", CSRC,
           os.path.join(ROOT, "tests", "offload_host_check.cpp"),
           os.path.join(CSRC, "zero_offload.cpp"), "-o", exe]
    build = subprocess.run(cmd, capture_output=True, text=True)
    if build.returncode != 0:
        pytest.fail("build failed:\n" + build.stderr[-4000:])
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("ok")
