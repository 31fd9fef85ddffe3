"""Seeded inputs placed into flat buffers (host arrays or device memory).

A stream's values are indexed by the global flat index of the partition; padding
elements (the tail of each unit up to a multiple of N_d) are zero.  Nothing here
computes any part of the optimizer step.
"""
from __future__ import annotations

import numpy as np

from . import Stream


def unit_parts(units, lo: int, hi: int):
    """Split [lo, hi) of the global flat space into (a, e, real) pieces (real = inside a
    tensor, else unit padding).  units: rows (first, count, numel, numel_pad, shard, base,
    shard_base) of the partition's unit table."""
    out = []
    for (_f, _c, numel, numel_pad, _s, base, _sb) in units:
        for a, e, real in ((base, base + numel, True), (base + numel, base + numel_pad, False)):
            a2, e2 = max(a, lo), min(e, hi)
            if a2 < e2:
                out.append((a2, e2, real))
    return out


def fill_device(dst, stream: Stream, units, lo: int, hi: int) -> None:
    """dst[j] = stream value at flat index lo + j, zero in padding (dst: an int16 CUDA
    tensor of at least hi - lo elements; filled on torch's current stream)."""
    import torch
    assert dst.numel() >= hi - lo and dst.dtype == torch.int16
    cs = torch.cuda.current_stream().cuda_stream
    for a, e, real in unit_parts(units, lo, hi):
        if real:
            stream.device(dst.data_ptr() + 2 * (a - lo), a, e - a, cs)
        else:
            dst[a - lo:e - lo].zero_()


def fill_host(stream: Stream, units, lo: int, hi: int) -> np.ndarray:
    """Host array of the stream's values at flat indices [lo, hi), zero in padding."""
    out = np.zeros(hi - lo, dtype=np.uint16)
    for a, e, real in unit_parts(units, lo, hi):
        if real:
            stream.host_into(out[a - lo:e - lo], a)
    return out


def values_at(stream: Stream, units, idx: np.ndarray) -> np.ndarray:
    """Stream values at flat indices idx (zero at padding)."""
    out = stream.at(idx)
    real = np.zeros(idx.size, dtype=bool)
    for (_f, _c, numel, _np, _s, base, _sb) in units:
        real |= (idx >= base) & (idx < base + numel)
    out[~real] = 0
    return out
