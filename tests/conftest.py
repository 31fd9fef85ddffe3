import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_sessionstart(session):
    """Build libzero.so in-tree when it is missing or older than its sources (a fresh checkout);
    the binding itself never builds and has no fallback."""
    import glob
    from zero_sharded_mixed_03_gb300 import _build
    srcs = glob.glob(os.path.join(_build.CSRC, "*")) + [os.path.join(ROOT, "include", "zero.h")]
    lib = _build.LIB
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs):
        _build.build()
