"""CPU oracle of the sharded mixed-precision AdamW step -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never does, and this
package never imports the product.  The arithmetic lives in
``zero_oracle.cpp`` (single-threaded C++17, -O2 -ffp-contract=off); this file
only marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "liboracle.so")
SRC = os.path.join(_HERE, "zero_oracle.cpp")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17"]

_lib = None
i64 = ctypes.c_int64
vp = ctypes.c_void_p


def build() -> str:
    # compile to a private file, then rename: a process loading the library never sees a
    # half-written file even when several processes build at once
    tmp = f"{LIB}.{os.getpid()}.tmp"
    cmd = ["g++", *CFLAGS, "-shared", "-fPIC", SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        L = ctypes.CDLL(LIB)
        L.orc_widen16.restype = ctypes.c_float
        L.orc_widen16.argtypes = [ctypes.c_uint16, ctypes.c_int]
        L.orc_round16.restype = ctypes.c_uint16
        L.orc_round16.argtypes = [ctypes.c_float, ctypes.c_int]
        L.orc_widen16_array.argtypes = [vp, i64, ctypes.c_int, vp]
        L.orc_round16_array.argtypes = [vp, i64, ctypes.c_int, vp]
        L.orc_consts.argtypes = [ctypes.c_double] * 5 + [i64, ctypes.c_double, ctypes.c_int, vp]
        L.orc_reduce.restype = ctypes.c_int
        L.orc_reduce.argtypes = [i64, ctypes.c_int, vp, ctypes.c_int, ctypes.c_float, vp]
        L.orc_adamw.argtypes = [i64, vp, vp, vp, vp, vp, ctypes.c_int, vp]
        L.orc_recast.argtypes = [i64, vp, ctypes.c_int, vp]
        L.orc_layout.restype = i64
        L.orc_layout.argtypes = [vp, i64, vp, i64, ctypes.c_int, vp, vp, i64]
        L.orc_shard_segments.restype = i64
        L.orc_shard_segments.argtypes = [vp, i64, vp, i64, ctypes.c_int, vp, i64]
        L.orc_bucket_segments.restype = i64
        L.orc_bucket_segments.argtypes = [i64, ctypes.c_int, i64, vp, i64]
        L.orc_memory.argtypes = [i64, ctypes.c_int, vp]
        L.orc_comm.argtypes = [i64, ctypes.c_int, vp]
        L.orc_sharded_step.restype = ctypes.c_int
        L.orc_sharded_step.argtypes = [vp, i64, vp, i64, ctypes.c_int, ctypes.c_int, i64,
                                       ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp]
        L.orc_sharded_step_ex.restype = ctypes.c_int
        L.orc_sharded_step_ex.argtypes = [vp, i64, vp, i64, ctypes.c_int, ctypes.c_int, i64,
                                          ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.c_double, ctypes.POINTER(ctypes.c_double)]
        L.orc_clip_coef.restype = ctypes.c_float
        L.orc_clip_coef.argtypes = [ctypes.c_double, ctypes.c_double]
        L.orc_pp_chunks.restype = i64
        L.orc_pp_chunks.argtypes = [vp, vp, i64, vp, i64, ctypes.c_int, vp, i64,
                                    ctypes.POINTER(i64)]
        L.orc_pp_step.restype = ctypes.c_int
        L.orc_pp_step.argtypes = [vp, vp, i64, vp, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                  vp, vp, vp, vp]
        L.orc_pp_step_ex.restype = ctypes.c_int
        L.orc_pp_step_ex.argtypes = [vp, vp, i64, vp, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                     vp, vp, vp, vp, ctypes.c_double, ctypes.POINTER(ctypes.c_double)]
        L.orc_pp_gather.restype = ctypes.c_int
        L.orc_pp_gather.argtypes = [vp, vp, i64, vp, i64, ctypes.c_int, i64, vp, vp]
        L.orc_scaler_update.restype = i64
        L.orc_scaler_update.argtypes = [ctypes.c_int, i64, ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(i64), ctypes.c_double, ctypes.c_double, i64,
                                        ctypes.c_double]
        L.orc_ddp_step.restype = ctypes.c_int
        L.orc_ddp_step.argtypes = [i64, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp, vp, vp]
        L.orc_gather_unit.restype = ctypes.c_int
        L.orc_gather_unit.argtypes = [vp, i64, vp, i64, ctypes.c_int, i64, vp, vp]
        _lib = L
    return _lib


# --------------------------------------------------------------------------- helpers

def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _ptrs(arrs: Sequence[Optional[np.ndarray]]):
    arr = (ctypes.c_void_p * max(1, len(arrs)))()
    for i, a in enumerate(arrs):
        arr[i] = None if a is None else a.ctypes.data
    return arr


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def widen16(h: np.ndarray, is_fp16: int) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.size, dtype=np.float32)
    lib().orc_widen16_array(_p(h), h.size, is_fp16, _p(out))
    return out.reshape(h.shape)


def round16(f: np.ndarray, is_fp16: int) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.size, dtype=np.uint16)
    lib().orc_round16_array(_p(f), f.size, is_fp16, _p(out))
    return out.reshape(f.shape)


def consts(hyper, t: int, loss_scale: float, n_d: int) -> np.ndarray:
    out = np.empty(9, dtype=np.float32)
    lib().orc_consts(hyper.lr, hyper.beta1, hyper.beta2, hyper.eps, hyper.weight_decay, t,
                     loss_scale, n_d, _p(out))
    return out


def reduce(contribs: Sequence[np.ndarray], is_fp16: int, inv: float):
    n = contribs[0].size
    g = np.empty(n, dtype=np.float32)
    flag = lib().orc_reduce(n, len(contribs), _ptrs(contribs), is_fp16, inv, _p(g))
    return g, flag


def adamw(g, p, m, v, k9, is_fp16, out16=None):
    """In place on p, m, v (float32 arrays); writes out16 when given."""
    lib().orc_adamw(g.size, _p(g), _p(p), _p(m), _p(v), _p(k9), is_fp16, _p(out16))


def recast(p, is_fp16, out16):
    lib().orc_recast(p.size, _p(p), is_fp16, _p(out16))


class Layout:
    """Oracle partition tables of one plan."""

    def __init__(self, sizes, n_d: int, unit_first=None):
        self.sizes = _i64(sizes)
        self.unit_first = None if not unit_first else _i64(unit_first)
        self.n_units_arg = 0 if self.unit_first is None else self.unit_first.size
        self.n_d = n_d
        nt = self.sizes.size
        cap = max(1, self.n_units_arg)
        self.tensor_offset = np.zeros(max(1, nt), dtype=np.int64)
        rows = np.zeros((cap, 7), dtype=np.int64)
        nu = lib().orc_layout(_p(self.sizes), nt, _p(self.unit_first), self.n_units_arg, n_d,
                              _p(self.tensor_offset), _p(rows), cap)
        if nu < 0:
            raise ValueError("invalid layout arguments")
        self.tensor_offset = self.tensor_offset[:nt]
        self.units = rows[:nu]          # first, count, numel, numel_pad, shard, base, shard_base
        self.total_pad = int(self.units[:, 3].sum())
        self.shard_total = int(self.units[:, 4].sum())

    def shard_segments(self) -> np.ndarray:
        L = lib()
        n = L.orc_shard_segments(_p(self.sizes), self.sizes.size, _p(self.unit_first),
                                 self.n_units_arg, self.n_d, None, 0)
        rows = np.zeros((max(1, n), 6), dtype=np.int64)
        L.orc_shard_segments(_p(self.sizes), self.sizes.size, _p(self.unit_first),
                             self.n_units_arg, self.n_d, _p(rows), n)
        return rows[:n]

    def bucket_segments(self, bucket_elems: int) -> np.ndarray:
        L = lib()
        n = L.orc_bucket_segments(self.total_pad, self.n_d, bucket_elems, None, 0)
        if n < 0:
            raise ValueError("invalid bucket arguments")
        rows = np.zeros((max(1, n), 5), dtype=np.int64)
        L.orc_bucket_segments(self.total_pad, self.n_d, bucket_elems, _p(rows), n)
        return rows[:n]


class PerParam:
    """Oracle of FSDP-2 per-parameter (dim-0) sharding."""

    def __init__(self, sizes, dim0, n_d: int, unit_first=None):
        self.sizes, self.dim0 = _i64(sizes), _i64(dim0)
        self.unit_first = None if not unit_first else _i64(unit_first)
        self.n_units_arg = 0 if self.unit_first is None else self.unit_first.size
        self.n_d = n_d
        L = lib()
        per = i64(0)
        n = L.orc_pp_chunks(_p(self.sizes), _p(self.dim0), self.sizes.size, _p(self.unit_first),
                            self.n_units_arg, n_d, None, 0, ctypes.byref(per))
        if n < 0:
            raise ValueError("invalid per-parameter layout")
        rows = np.zeros((max(1, n), 9), dtype=np.int64)
        L.orc_pp_chunks(_p(self.sizes), _p(self.dim0), self.sizes.size, _p(self.unit_first),
                        self.n_units_arg, n_d, _p(rows), n, None)
        self.chunks = rows[:n]       # rank, unit, tensor, row0, rows, cols, c_rows, contrib_off, state_off
        self.per_rank = per.value
        firsts = list(self.unit_first) if self.unit_first is not None else [0]
        ends = firsts[1:] + [self.sizes.size]
        self.unit_numel = [int(self.sizes[f:e].sum()) for f, e in zip(firsts, ends)]
        self.unit_base = np.concatenate([[0], np.cumsum(self.unit_numel)]).astype(np.int64)

    def step(self, is_fp16, contribs, bound, p, m, v, shard16, k9) -> int:
        bound = np.ascontiguousarray(np.asarray(bound, dtype=np.int32))
        return lib().orc_pp_step(_p(self.sizes), _p(self.dim0), self.sizes.size, _p(self.unit_first),
                                 self.n_units_arg, self.n_d, is_fp16, _ptrs(contribs), _p(bound),
                                 _ptrs(p), _ptrs(m), _ptrs(v), _ptrs(shard16), _p(k9))

    def step_ex(self, is_fp16, contribs, bound, p, m, v, shard16, k9, max_norm: float):
        """step with the global gradient norm (R8): returns (flag, norm^2); max_norm > 0 clips."""
        bound = np.ascontiguousarray(np.asarray(bound, dtype=np.int32))
        norm2 = ctypes.c_double(0.0)
        flag = lib().orc_pp_step_ex(_p(self.sizes), _p(self.dim0), self.sizes.size, _p(self.unit_first),
                                    self.n_units_arg, self.n_d, is_fp16, _ptrs(contribs), _p(bound),
                                    _ptrs(p), _ptrs(m), _ptrs(v), _ptrs(shard16), _p(k9),
                                    float(max_norm), ctypes.byref(norm2))
        return flag, norm2.value

    def gather(self, unit: int, shard16) -> np.ndarray:
        out = np.zeros(self.unit_numel[unit], dtype=np.uint16)
        rc = lib().orc_pp_gather(_p(self.sizes), _p(self.dim0), self.sizes.size, _p(self.unit_first),
                                 self.n_units_arg, self.n_d, unit, _ptrs(shard16), _p(out))
        if rc != 0:
            raise ValueError("invalid gather arguments")
        return out


def memory(phi_pad: int, n_d: int) -> np.ndarray:
    out = np.zeros(15, dtype=np.int64)
    lib().orc_memory(phi_pad, n_d, _p(out))
    return out


def comm(phi_pad: int, n_d: int) -> np.ndarray:
    out = np.zeros(4, dtype=np.int64)
    lib().orc_comm(phi_pad, n_d, _p(out))
    return out


def sharded_step(layout: Layout, stage: int, bucket_elems: int, is_fp16: int, contribs, bound,
                 p, m, v, shard16, full16, k9) -> int:
    bound = np.ascontiguousarray(np.asarray(bound, dtype=np.int32))
    n_d = layout.n_d
    return lib().orc_sharded_step(
        _p(layout.sizes), layout.sizes.size, _p(layout.unit_first), layout.n_units_arg, n_d,
        stage, bucket_elems, is_fp16, _ptrs(contribs), _p(bound), _ptrs(p), _ptrs(m), _ptrs(v),
        _ptrs(shard16 if shard16 is not None else [None] * n_d), _p(full16), _p(k9))


class ScalerState:
    """Oracle-side loss-scale trajectory (scale, clean-step counter, applied steps t)."""

    def __init__(self, scaler_cfg, t: int = 0):
        self.cfg = scaler_cfg
        self.scale = scaler_cfg.init_scale if scaler_cfg is not None else 1.0
        self.good = 0
        self.t = t

    def update(self, flag: int) -> None:
        if self.cfg is None:
            self.t = self.t if flag else self.t + 1
            return
        sc = ctypes.c_double(self.scale)
        gd = ctypes.c_int64(self.good)
        self.t = int(lib().orc_scaler_update(int(flag), self.t, ctypes.byref(sc), ctypes.byref(gd),
                                             self.cfg.growth_factor, self.cfg.backoff_factor,
                                             self.cfg.growth_interval, self.cfg.min_scale))
        self.scale, self.good = sc.value, gd.value


def sharded_step_ex(layout: Layout, stage: int, bucket_elems: int, is_fp16: int, contribs,
                    bound, p, m, v, shard16, full16, k9, max_norm: float = 0.0):
    """Sharded step with the optional norm / clipping; returns (flag, norm^2)."""
    bound = np.ascontiguousarray(np.asarray(bound, dtype=np.int32))
    n_d = layout.n_d
    norm2 = ctypes.c_double(0.0)
    flag = lib().orc_sharded_step_ex(
        _p(layout.sizes), layout.sizes.size, _p(layout.unit_first), layout.n_units_arg, n_d,
        stage, bucket_elems, is_fp16, _ptrs(contribs), _p(bound), _ptrs(p), _ptrs(m), _ptrs(v),
        _ptrs(shard16 if shard16 is not None else [None] * n_d), _p(full16), _p(k9),
        float(max_norm), ctypes.byref(norm2))
    return flag, norm2.value


def clip_coef(norm2: float, max_norm: float) -> float:
    return float(lib().orc_clip_coef(norm2, max_norm))


def ddp_step(contribs, is_fp16, p, m, v, out16, k9) -> int:
    return lib().orc_ddp_step(p.size, len(contribs), _ptrs(contribs), is_fp16, _p(p), _p(m),
                              _p(v), _p(out16), _p(k9))


def gather_unit(layout: Layout, unit: int, shard16) -> np.ndarray:
    U = layout.units[unit]
    out = np.zeros(int(U[3]), dtype=np.uint16)
    rc = lib().orc_gather_unit(_p(layout.sizes), layout.sizes.size, _p(layout.unit_first),
                               layout.n_units_arg, layout.n_d, unit, _ptrs(shard16), _p(out))
    if rc != 0:
        raise ValueError("invalid gather arguments")
    return out
