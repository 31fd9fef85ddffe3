"""Python binding of libzero (the sharded mixed-precision AdamW step for GB300).

Thin ctypes marshalling over the C ABI declared in ``include/zero.h``: every
function has the C name and forwards plain integers (device pointers, sizes,
stream handles).  All arithmetic runs in the CUDA kernels of ``libzero.so``;
there is no Python or CPU fallback.  If the library has not been built, import
succeeds but the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libzero.so")

ZERO_OK, ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA, ZERO_ESTATE, ZERO_ERANGE, ZERO_ETIMEOUT, ZERO_ENOMEM = range(8)
ZERO_BF16, ZERO_FP16 = 0, 1
ZERO_MAX_RANKS = 128
ZERO_REPORT_GRAD_NORM = 1
(ZERO_OPT_STAGING, ZERO_OPT_WAIT_LIMIT_NS, ZERO_OPT_BULK_TILE, ZERO_OPT_BULK_STAGES,
 ZERO_OPT_LAST_STEP_KERNEL, ZERO_OPT_GATHER_STAGING, ZERO_OPT_GATHER_CHUNK,
 ZERO_OPT_GATHER_STAGES, ZERO_OPT_HOST_PIPELINE, ZERO_OPT_HOST_H2D_BYTES,
 ZERO_OPT_HOST_D2H_BYTES, ZERO_OPT_LAST_GATHER_IN_STEP, ZERO_OPT_OFFLOAD_DEFER,
 ZERO_OPT_UNIT_ORDER) = range(14)
ZERO_STAGING_REGISTER_LOADS, ZERO_STAGING_BULK, ZERO_STAGING_AUTO = range(3)
(ZERO_TABLE_TENSOR_OFFSET, ZERO_TABLE_UNITS, ZERO_TABLE_SHARD_SEGMENTS,
 ZERO_TABLE_BUCKET_SEGMENTS, ZERO_TABLE_STATE_LAYOUT, ZERO_TABLE_PARAM_CHUNKS) = range(6)
TABLE_COLS = {0: 1, 1: 7, 2: 6, 3: 5, 4: 4, 5: 10}
STATUS_NAMES = {0: "ZERO_OK", 1: "ZERO_EINVAL", 2: "ZERO_EALIGN", 3: "ZERO_ECUDA",
                4: "ZERO_ESTATE", 5: "ZERO_ERANGE", 6: "ZERO_ETIMEOUT", 7: "ZERO_ENOMEM"}

EXPORTED = ["zero_plan_create", "zero_plan_create_per_param", "zero_plan_info", "zero_rank_state_elems", "zero_plan_tables",
            "zero_bind", "zero_bind_peer", "zero_step", "zero_step_finish", "zero_gather_layer",
            "zero_release_layer", "zero_memory_report", "zero_comm_report", "zero_set_scaler",
            "zero_read_state", "zero_restore_state", "zero_grad_norm",
            "zero_step_units_overlapped", "zero_bind_offload", "zero_offload_step",
            "zero_offload_finish", "zero_set_option", "zero_get_option",
            "zero_bind_host_staging", "zero_step_host", "zero_step_host_finish", "zero_grad_norm_host",
            "zero_step_gather_next",
            "zero_last_error", "zero_plan_destroy", "zero_step_range_noalloc"]
ZERO_NOALLOC_SCRATCH_BYTES = 256


class ZeroError(RuntimeError):
    def __init__(self, status: int, msg: str, result=None):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status
        self.result = result   # the step state read with a ZERO_ETIMEOUT report


class zero_hyper_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("max_grad_norm", ctypes.c_double), ("flags", ctypes.c_int64)]


class zero_scaler_t(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_double), ("growth_factor", ctypes.c_double),
                ("backoff_factor", ctypes.c_double), ("min_scale", ctypes.c_double),
                ("growth_interval", ctypes.c_int64), ("good_steps", ctypes.c_int64)]


class zero_plan_info_t(ctypes.Structure):
    _fields_ = [("n_tensors", ctypes.c_int64), ("n_units", ctypes.c_int64),
                ("n_buckets", ctypes.c_int64), ("phi", ctypes.c_int64),
                ("phi_pad", ctypes.c_int64), ("shard", ctypes.c_int64),
                ("max_contrib_elems", ctypes.c_int64), ("max_unit_pad", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("n_d", ctypes.c_int32),
                ("stage", ctypes.c_int32), ("dtype16", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("host_staging_bytes", ctypes.c_int64)]


class zero_step_result_t(ctypes.Structure):
    _fields_ = [("skipped", ctypes.c_int32), ("current", ctypes.c_int32),
                ("t", ctypes.c_int64), ("scale", ctypes.c_double),
                ("good_steps", ctypes.c_int64), ("skipped_total", ctypes.c_int64),
                ("finished", ctypes.c_int64), ("grad_norm", ctypes.c_double)]


class zero_mem_report_t(ctypes.Structure):
    _fields_ = [("logical", (ctypes.c_int64 * 3) * 4), ("logical_total", ctypes.c_int64 * 4),
                ("logical_ddp_fp32_grads", ctypes.c_int64),
                ("physical_state_bytes", ctypes.c_int64),
                ("physical_param16_bytes", ctypes.c_int64),
                ("physical_contrib_bytes", ctypes.c_int64),
                ("physical_gather_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]


class zero_comm_report_t(ctypes.Structure):
    _fields_ = [("per_collective", ctypes.c_int64), ("ddp", ctypes.c_int64),
                ("zero1", ctypes.c_int64), ("zero2", ctypes.c_int64), ("zero3", ctypes.c_int64),
                ("this_stage", ctypes.c_int64), ("bytes_per_elem", ctypes.c_int64),
                ("collectives_per_step", ctypes.c_int64)]


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def lib() -> ctypes.CDLL:
    """Load libzero.so; raises if it is missing (no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libzero.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        st = _int
        L.zero_plan_create.restype = st
        L.zero_plan_create.argtypes = [_vp, _i64, _int, _int, _i64, _vp, _i64, _int,
                                       ctypes.POINTER(_vp)]
        L.zero_plan_create_per_param.restype = st
        L.zero_plan_create_per_param.argtypes = [_vp, _vp, _i64, _int, _vp, _i64, _int,
                                                 ctypes.POINTER(_vp)]
        L.zero_plan_info.restype = st
        L.zero_plan_info.argtypes = [_vp, ctypes.POINTER(zero_plan_info_t)]
        L.zero_rank_state_elems.restype = st
        L.zero_rank_state_elems.argtypes = [_vp, _int, ctypes.POINTER(_i64)]
        L.zero_plan_tables.restype = st
        L.zero_plan_tables.argtypes = [_vp, _int, _vp, _i64, ctypes.POINTER(_i64)]
        L.zero_bind.restype = st
        L.zero_bind.argtypes = [_vp, _int, _vp, _vp, _vp, _vp, _vp, _vp]
        L.zero_bind_peer.restype = st
        L.zero_bind_peer.argtypes = [_vp, _int, _vp]
        L.zero_step.restype = st
        L.zero_step.argtypes = [_vp, _vp, _i64, _i64, ctypes.POINTER(zero_hyper_t), _vp]
        L.zero_step_finish.restype = st
        L.zero_step_finish.argtypes = [_vp, _vp, ctypes.POINTER(zero_step_result_t)]
        L.zero_set_scaler.restype = st
        L.zero_set_scaler.argtypes = [_vp, ctypes.POINTER(zero_scaler_t), _vp]
        L.zero_read_state.restype = st
        L.zero_read_state.argtypes = [_vp, _vp, ctypes.POINTER(zero_step_result_t)]
        L.zero_step_units_overlapped.restype = st
        L.zero_step_units_overlapped.argtypes = [_vp, _vp, _i64, _vp, ctypes.POINTER(zero_hyper_t),
                                                 _vp, _vp, ctypes.POINTER(zero_step_result_t)]
        L.zero_bind_offload.restype = st
        L.zero_bind_offload.argtypes = [_vp, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.zero_offload_step.restype = st
        L.zero_offload_step.argtypes = [_vp, _vp, _i64, _i64, ctypes.POINTER(zero_hyper_t), _vp]
        L.zero_offload_finish.restype = st
        L.zero_offload_finish.argtypes = [_vp, _int, _vp, ctypes.POINTER(zero_step_result_t)]
        L.zero_step_gather_next.restype = st
        L.zero_step_gather_next.argtypes = [_vp, _vp, _i64, _i64, ctypes.POINTER(zero_hyper_t), _i64,
                                            _vp, _vp]
        L.zero_bind_host_staging.restype = st
        L.zero_bind_host_staging.argtypes = [_vp, _vp, _i64]
        L.zero_step_host.restype = st
        L.zero_step_host.argtypes = [_vp, _vp, _i64, _i64, ctypes.POINTER(zero_hyper_t), _vp, _vp]
        L.zero_grad_norm_host.restype = st
        L.zero_grad_norm_host.argtypes = [_vp, _vp, _i64, _i64, _vp]
        L.zero_step_host_finish.restype = st
        L.zero_step_host_finish.argtypes = [_vp, _vp, ctypes.POINTER(zero_step_result_t)]
        L.zero_grad_norm.restype = st
        L.zero_grad_norm.argtypes = [_vp, _vp, _i64, _i64, _vp]
        L.zero_set_option.restype = st
        L.zero_set_option.argtypes = [_vp, _int, _i64]
        L.zero_get_option.restype = st
        L.zero_get_option.argtypes = [_vp, _int, ctypes.POINTER(_i64)]
        L.zero_restore_state.restype = st
        L.zero_restore_state.argtypes = [_vp, ctypes.POINTER(zero_step_result_t), _vp]
        L.zero_gather_layer.restype = st
        L.zero_gather_layer.argtypes = [_vp, _i64, _vp, _vp]
        L.zero_release_layer.restype = st
        L.zero_release_layer.argtypes = [_vp, _i64]
        L.zero_memory_report.restype = st
        L.zero_memory_report.argtypes = [_vp, ctypes.POINTER(zero_mem_report_t)]
        L.zero_comm_report.restype = st
        L.zero_comm_report.argtypes = [_vp, ctypes.POINTER(zero_comm_report_t)]
        L.zero_last_error.restype = ctypes.c_char_p
        L.zero_last_error.argtypes = []
        L.zero_step_range_noalloc.restype = st
        L.zero_step_range_noalloc.argtypes = [_vp, _int, _i64, _int, _vp, _vp, _vp, _vp, _vp, _vp,
                                              _vp, ctypes.POINTER(zero_hyper_t), _i64,
                                              ctypes.c_double, _vp, ctypes.POINTER(ctypes.c_int32)]
        L.zero_plan_destroy.restype = None
        L.zero_plan_destroy.argtypes = [_vp]
        _lib = L
    return _lib


def _check(status: int, result=None) -> None:
    if status != ZERO_OK:
        msg = lib().zero_last_error()
        raise ZeroError(status, msg.decode() if msg else "", result)


def _ptr_array(ptrs: Sequence[Optional[int]]):
    arr = (_vp * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = p or None
    return arr


def _i64_array(vals: Sequence[int]):
    arr = (_i64 * max(1, len(vals)))()
    for i, v in enumerate(vals):
        arr[i] = int(v)
    return arr


# --------------------------------------------------------------------------- C-named calls

def zero_plan_create(tensor_sizes: Sequence[int], n_d: int, stage: int, bucket_elems: int = 0,
                     unit_first: Optional[Sequence[int]] = None, dtype16: int = ZERO_BF16) -> int:
    sizes = _i64_array(tensor_sizes)
    units = _i64_array(unit_first) if unit_first else None
    out = _vp()
    _check(lib().zero_plan_create(sizes, len(tensor_sizes), n_d, stage, bucket_elems, units,
                                  len(unit_first) if unit_first else 0, dtype16,
                                  ctypes.byref(out)))
    return int(out.value)


def zero_plan_create_per_param(tensor_sizes: Sequence[int], dim0: Sequence[int], n_d: int,
                               unit_first: Optional[Sequence[int]] = None,
                               dtype16: int = ZERO_BF16) -> int:
    sizes = _i64_array(tensor_sizes)
    d0 = _i64_array(dim0)
    units = _i64_array(unit_first) if unit_first else None
    out = _vp()
    _check(lib().zero_plan_create_per_param(sizes, d0, len(tensor_sizes), n_d, units,
                                            len(unit_first) if unit_first else 0, dtype16,
                                            ctypes.byref(out)))
    return int(out.value)


def zero_plan_info(plan: int) -> zero_plan_info_t:
    info = zero_plan_info_t()
    _check(lib().zero_plan_info(plan, ctypes.byref(info)))
    return info


def zero_rank_state_elems(plan: int, rank: int) -> int:
    n = _i64()
    _check(lib().zero_rank_state_elems(plan, rank, ctypes.byref(n)))
    return int(n.value)


def zero_plan_tables(plan: int, which: int):
    """Returns a list of rows (tuples of ints)."""
    n = _i64()
    _check(lib().zero_plan_tables(plan, which, None, 0, ctypes.byref(n)))
    cols = TABLE_COLS[which]
    buf = (_i64 * max(1, n.value * cols))()
    _check(lib().zero_plan_tables(plan, which, buf, n.value * cols, ctypes.byref(n)))
    return [tuple(buf[i * cols:(i + 1) * cols]) for i in range(n.value)]


def zero_bind(plan: int, rank: int, master: Sequence[int], m: Sequence[int], v: Sequence[int],
              shard16: Optional[int], full16: Optional[int], workspace: int) -> None:
    _check(lib().zero_bind(plan, rank, _ptr_array(master), _ptr_array(m), _ptr_array(v),
                           shard16 or None, full16 or None, workspace or None))


def zero_bind_peer(plan: int, rank: int, shard16: int) -> None:
    _check(lib().zero_bind_peer(plan, rank, shard16 or None))


def zero_set_scaler(plan: int, scaler: Optional[zero_scaler_t], stream: int = 0) -> None:
    _check(lib().zero_set_scaler(plan, ctypes.byref(scaler) if scaler is not None else None,
                                 stream or None))


def zero_step(plan: int, grad_contribs: Sequence[int], which: int, hyper: zero_hyper_t,
              stream: int = 0) -> None:
    _check(lib().zero_step(plan, _ptr_array(grad_contribs), len(grad_contribs), which,
                           ctypes.byref(hyper), stream or None))


def zero_step_gather_next(plan: int, grad_contribs: Sequence[int], unit: int, hyper: zero_hyper_t,
                          next_unit: int, next_full16: int, stream: int = 0) -> None:
    _check(lib().zero_step_gather_next(plan, _ptr_array(grad_contribs), len(grad_contribs), unit,
                                       ctypes.byref(hyper), next_unit, next_full16 or None,
                                       stream or None))


def zero_grad_norm(plan: int, grad_contribs: Sequence[int], which: int, stream: int = 0) -> None:
    _check(lib().zero_grad_norm(plan, _ptr_array(grad_contribs), len(grad_contribs), which,
                                stream or None))


def zero_step_units_overlapped(plan: int, unit_contribs: Sequence[int], gather_bufs: Sequence[int],
                               hyper: zero_hyper_t, compute_stream: int, comm_stream: Optional[int],
                               wait: bool = True) -> Optional[zero_step_result_t]:
    """comm_stream None / 0: the one-stream schedule (unit u+1's gather inside unit u's step)."""
    res = zero_step_result_t() if wait else None
    _check(lib().zero_step_units_overlapped(plan, _ptr_array(unit_contribs), len(unit_contribs),
                                            _ptr_array(gather_bufs), ctypes.byref(hyper),
                                            compute_stream or None, comm_stream or None,
                                            ctypes.byref(res) if res is not None else None))
    return res


def zero_bind_offload(plan: int, rank: int, master: int, m: int, v: int, grad_host: int,
                      param16_host: int, shard16: Optional[int], full16: Optional[int],
                      workspace: int) -> None:
    _check(lib().zero_bind_offload(plan, rank, master or None, m or None, v or None,
                                   grad_host or None, param16_host or None, shard16 or None,
                                   full16 or None, workspace or None))


def zero_offload_step(plan: int, grad_contribs: Sequence[int], which: int, hyper: zero_hyper_t,
                      stream: int = 0) -> None:
    _check(lib().zero_offload_step(plan, _ptr_array(grad_contribs), len(grad_contribs), which,
                                   ctypes.byref(hyper), stream or None))


def zero_offload_finish(plan: int, threads: int, stream: int = 0,
                        wait: bool = True) -> Optional[zero_step_result_t]:
    res = zero_step_result_t() if wait else None
    _check(lib().zero_offload_finish(plan, threads, stream or None,
                                     ctypes.byref(res) if res is not None else None))
    return res


def zero_bind_host_staging(plan: int, staging: Sequence[int], bytes_each: int) -> None:
    _check(lib().zero_bind_host_staging(plan, _ptr_array(staging), bytes_each))


def zero_step_host(plan: int, host_contribs: Sequence[int], which: int, hyper: zero_hyper_t,
                   host_out16: int, stream: int = 0) -> None:
    _check(lib().zero_step_host(plan, _ptr_array(host_contribs), len(host_contribs), which,
                                ctypes.byref(hyper), host_out16 or None, stream or None))


def zero_grad_norm_host(plan: int, host_contribs: Sequence[int], which: int, stream: int = 0) -> None:
    _check(lib().zero_grad_norm_host(plan, _ptr_array(host_contribs), len(host_contribs), which,
                                     stream or None))


def zero_step_host_finish(plan: int, stream: int = 0) -> zero_step_result_t:
    """End a step that had zero_step_host calls (synchronises); returns the step state."""
    res = zero_step_result_t()
    _check(lib().zero_step_host_finish(plan, stream or None, ctypes.byref(res)), res)
    return res


def zero_step_finish(plan: int, stream: int = 0, wait: bool = True) -> Optional[zero_step_result_t]:
    """Enqueue the commit; with wait=True also read back the step state (synchronises)."""
    res = zero_step_result_t() if wait else None
    _check(lib().zero_step_finish(plan, stream or None,
                                  ctypes.byref(res) if res is not None else None), res)
    return res


def zero_restore_state(plan: int, state: zero_step_result_t, stream: int = 0) -> None:
    _check(lib().zero_restore_state(plan, ctypes.byref(state), stream or None))


def zero_read_state(plan: int, stream: int = 0) -> zero_step_result_t:
    res = zero_step_result_t()
    _check(lib().zero_read_state(plan, stream or None, ctypes.byref(res)), res)
    return res


def zero_set_option(plan: int, option: int, value: int) -> None:
    """ZERO_OPT_STAGING (ZERO_STAGING_REGISTER_LOADS / _BULK / _AUTO), ZERO_OPT_WAIT_LIMIT_NS,
    ZERO_OPT_BULK_TILE, ZERO_OPT_BULK_STAGES (0 = chosen from N_d); the gather's
    ZERO_OPT_GATHER_STAGING, ZERO_OPT_GATHER_CHUNK, ZERO_OPT_GATHER_STAGES (0 = default);
    ZERO_OPT_HOST_PIPELINE (host-buffer steps: 1 pipelined, 0 serial)."""
    _check(lib().zero_set_option(plan, option, int(value)))


def zero_get_option(plan: int, option: int) -> int:
    """An option's value in effect, or ZERO_OPT_LAST_STEP_KERNEL (1 staged, 0 register loads)."""
    v = _i64()
    _check(lib().zero_get_option(plan, option, ctypes.byref(v)))
    return v.value


def zero_gather_layer(plan: int, unit: int, full_unit16: int, stream: int = 0) -> None:
    _check(lib().zero_gather_layer(plan, unit, full_unit16 or None, stream or None))


def zero_release_layer(plan: int, unit: int) -> None:
    _check(lib().zero_release_layer(plan, unit))


def zero_memory_report(plan: int) -> zero_mem_report_t:
    rep = zero_mem_report_t()
    _check(lib().zero_memory_report(plan, ctypes.byref(rep)))
    return rep


def zero_comm_report(plan: int) -> zero_comm_report_t:
    rep = zero_comm_report_t()
    _check(lib().zero_comm_report(plan, ctypes.byref(rep)))
    return rep


def zero_last_error() -> str:
    msg = lib().zero_last_error()
    return msg.decode() if msg else ""


def zero_plan_destroy(plan: int) -> None:
    if plan:
        lib().zero_plan_destroy(plan)


def zero_step_range_noalloc(grad_contribs: Sequence[int], n: int, dtype16: int, master_in: int,
                            m_in: int, v_in: int, master_out: int, m_out: int, v_out: int,
                            out16: int, hyper: zero_hyper_t, t: int, loss_scale: float = 1.0,
                            stream: int = 0) -> int:
    """Fused step over one flat range without any workspace; returns the non-finite flag."""
    flag = ctypes.c_int32(0)
    _check(lib().zero_step_range_noalloc(_ptr_array(grad_contribs), len(grad_contribs), n, dtype16,
                                         master_in or None, m_in or None, v_in or None,
                                         master_out or None, m_out or None, v_out or None,
                                         out16 or None, ctypes.byref(hyper), t, loss_scale,
                                         stream or None, ctypes.byref(flag)))
    return int(flag.value)


def hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=0.0,
          report_grad_norm=False) -> zero_hyper_t:
    return zero_hyper_t(lr, beta1, beta2, eps, weight_decay, max_grad_norm,
                        ZERO_REPORT_GRAD_NORM if report_grad_norm else 0)


def scaler(scale=65536.0, growth_factor=2.0, backoff_factor=0.5, min_scale=1.0,
           growth_interval=1000, good_steps=0) -> zero_scaler_t:
    return zero_scaler_t(scale, growth_factor, backoff_factor, min_scale, growth_interval,
                         good_steps)
