"""The C ABI used from a C program, with no Python and no torch in the process: one ZeRO-2
step of 4 emulated ranks (tests/abi_from_c.c), device memory from the CUDA driver API on the
primary context, checked against the closed-form first AdamW step."""
import os
import shutil
import subprocess

import pytest
import torch

import zero_sharded_mixed_03_gb300 as Z

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_steps_through_the_abi(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    Z.lib()                                    # the library is built
    pkg = os.path.dirname(Z.LIB_PATH)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "abi_from_c")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", os.path.join(ROOT, "tests", "abi_from_c.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", pkg, "-lzero", f"-Wl,-rpath,{pkg}",
           "-L", os.path.join(cuda, "lib64", "stubs"), "-lcuda", "-lm", "-o", exe]
    build = subprocess.run(cmd, capture_output=True, text=True)
    assert build.returncode == 0, build.stderr[-4000:]
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("ok"), run.stdout + run.stderr
