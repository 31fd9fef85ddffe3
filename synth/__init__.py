"""Seeded synthetic inputs (Python side of the generator module).

Loads the host fill library (``libsynth_host.so``, gcc) and, when a GPU path is
used, the device fill library (``libsynth_dev.so``, nvcc sm_103a).  Both are
built from ``synth_core.h``, so the same stream gives the same bits on the
host and on the device.  This package only prepares inputs: it contains none
of the arithmetic of the optimizer step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
GENCODE = "arch=compute_103a,code=sm_103a"

_host = None
_dev = None

u64 = ctypes.c_uint64
i64 = ctypes.c_int64


def build_host() -> str:
    src = os.path.join(_HERE, "synth_host.cpp")
    tmp = f"{HOST_LIB}.{os.getpid()}.tmp"        # renamed into place: never half-written
    cmd = ["g++", "-O2", "-ffp-contract=off", "-std=c++17", "-shared", "-fPIC", src, "-o",
           tmp, "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_device() -> str:
    src = os.path.join(_HERE, "synth_dev.cu")
    tmp = f"{DEV_LIB}.{os.getpid()}.tmp"
    cmd = [NVCC, "-gencode", GENCODE, "-O3", "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
           src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, DEV_LIB)
    return DEV_LIB


def _load_host():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            build_host()
        lib = ctypes.CDLL(HOST_LIB)
        lib.syn_fill_host.restype = ctypes.c_int
        lib.syn_fill_host.argtypes = [ctypes.c_void_p, i64, i64, u64, u64, u64, u64, u64,
                                      ctypes.c_double, ctypes.c_int, ctypes.c_int, i64,
                                      ctypes.c_uint32, ctypes.c_int]
        lib.syn_values_at.restype = ctypes.c_int
        lib.syn_values_at.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, u64, u64, u64, u64,
                                      u64, ctypes.c_double, ctypes.c_int, ctypes.c_int, i64,
                                      ctypes.c_uint32]
        lib.syn_hash.restype = u64
        lib.syn_hash.argtypes = [u64]
        lib.syn_stream_key.restype = u64
        lib.syn_stream_key.argtypes = [u64, u64, u64, u64, u64]
        lib.syn_scale.restype = ctypes.c_float
        lib.syn_scale.argtypes = [ctypes.c_double]
        lib.syn_round_bf16.restype = ctypes.c_uint16
        lib.syn_round_bf16.argtypes = [ctypes.c_float]
        lib.syn_round_fp16.restype = ctypes.c_uint16
        lib.syn_round_fp16.argtypes = [ctypes.c_float]
        _host = lib
    return _host


def _load_dev():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(f"device generator library missing: {DEV_LIB} (run the build)")
        lib = ctypes.CDLL(DEV_LIB)
        lib.syn_fill_device.restype = ctypes.c_int
        lib.syn_fill_device.argtypes = [ctypes.c_void_p, i64, i64, u64, u64, u64, u64, u64,
                                        ctypes.c_double, ctypes.c_int, ctypes.c_int, i64,
                                        ctypes.c_uint32, ctypes.c_void_p]
        _dev = lib
    return _dev


def hash64(x: int) -> int:
    return int(_load_host().syn_hash(x & 0xFFFFFFFFFFFFFFFF))


def stream_key(seed: int, wid: int, kind: int, step: int, rank: int) -> int:
    return int(_load_host().syn_stream_key(seed, wid, kind, step, rank))


def scale_for_sigma(sigma: float) -> float:
    return float(_load_host().syn_scale(sigma))


class Stream:
    """One generator stream: (workload id, kind, step, rank) + value recipe."""

    def __init__(self, wid: int, kind: int, step: int, rank: int, sigma: float, dtype: int,
                 outliers: bool = False, inject_index: int = -1, inject_bits: int = 0,
                 seed: int = 0):
        self.args = (seed, wid, kind, step, rank, float(sigma), int(dtype), int(bool(outliers)),
                     int(inject_index), int(inject_bits))

    def host(self, start: int, n: int, threads: int = 0) -> np.ndarray:
        out = np.empty(n, dtype=np.uint16)
        rc = _load_host().syn_fill_host(out.ctypes.data, n, start, *self.args, threads)
        if rc != 0:
            raise RuntimeError(f"syn_fill_host failed ({rc})")
        return out

    def host_into(self, dst: np.ndarray, start: int, threads: int = 0) -> None:
        assert dst.dtype == np.uint16 and dst.flags.c_contiguous
        rc = _load_host().syn_fill_host(dst.ctypes.data, dst.size, start, *self.args, threads)
        if rc != 0:
            raise RuntimeError(f"syn_fill_host failed ({rc})")

    def at(self, idx: np.ndarray) -> np.ndarray:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.empty(idx.size, dtype=np.uint16)
        rc = _load_host().syn_values_at(out.ctypes.data, idx.ctypes.data, idx.size, *self.args)
        if rc != 0:
            raise RuntimeError(f"syn_values_at failed ({rc})")
        return out

    def device(self, ptr: int, start: int, n: int, stream: Optional[int] = None) -> None:
        rc = _load_dev().syn_fill_device(ctypes.c_void_p(ptr), n, start, *self.args,
                                          ctypes.c_void_p(stream or 0))
        if rc != 0:
            raise RuntimeError(f"syn_fill_device failed ({rc})")


def param_stream(w) -> Stream:
    from .workloads import KIND_PARAM
    return Stream(w.wid, KIND_PARAM, 0, 0, w.param_sigma, w.dtype)


def grad_stream(w, step: int, rank: int, planted: bool = True) -> Stream:
    """Gradient contribution of `rank` at 1-based `step`, over the global flat index space.

    planted=False leaves out the workload's planted inf (the values are otherwise identical).
    """
    from .workloads import KIND_GRAD, INF16
    inj_idx, inj_bits = -1, 0
    if planted and w.inject is not None and w.inject[0] == step and w.inject[1] == rank:
        inj_idx, inj_bits = w.inject[2], INF16[w.dtype]
    return Stream(w.wid, KIND_GRAD, step, rank, w.grad_sigma, w.dtype, w.outliers, inj_idx,
                  inj_bits)
