"""The C example in README.md compiles against include/zero.h (syntax and types only)."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_c_example_compiles(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```c\n(.*?)```", text, re.S)
    assert blocks, "README.md has no C example"
    src = tmp_path / "example.c"
    src.write_text(blocks[0])
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
