"""A synthetic workload bound to the product API on the GPU.

Run creates the emulated group (plan, fp32 state, 16-bit buffers and workspace through
libzero's C ABI), writes the seeded initial 16-bit parameters and their exact fp32 widening
into the master state, sets the workload's loss scaler, and reads results back.  It is the
input side shared by the benchmark and the GPU tests; it contains none of the optimizer
step's arithmetic and does not load the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import zero_sharded_mixed_03_gb300 as Z
from zero_sharded_mixed_03_gb300.emulate import EmulatedGroup

from . import grad_stream, param_stream
from . import workloads as W
from .fill import fill_device

TORCH16 = {W.BF16: torch.bfloat16, W.FP16: torch.float16}


class Run:
    """One workload on the GPU through the product API."""

    def __init__(self, w: W.Workload, bound=None, peers: bool = True, alloc_contribs: bool = True,
                 options=None):
        """options: {ZERO_OPT_*: value} applied with zero_set_option (e.g. bulk staging)."""
        self.w = w
        b = bound if bound is not None else w.ranks()
        self.g = EmulatedGroup(w.sizes, w.n_d, w.stage, w.bucket_elems, w.unit_first or None,
                               w.dtype, b, dim0=w.dim0 if w.per_param else None,
                               offload=w.offload)
        for opt, val in (options or {}).items():
            self.g.set_option(opt, val)
        self.units = self.g.units
        self.info = self.g.info
        self.bound = list(b)
        t16 = TORCH16[w.dtype]
        ps = param_stream(w)
        if w.stage != 3:
            fill_device(self.g.full16, ps, self.units, 0, int(self.info.phi_pad))
            S = self.units[0][4] if self.units else 0
            for r in self.bound:
                off = self.g.phys_off[r][0]
                self.g.state[r]["master"][0][off:off + S] = \
                    self.g.full16[r * S:(r + 1) * S].view(t16).float()
        elif w.per_param:
            ranks = list(range(w.n_d)) if peers else self.bound
            for r in ranks:
                sh = self.g.shard16[r] if r in self.g.shard16 else self.g.bind_peer_shard(r)
                for (_r, u, _t, _row0, rows, cols, c_rows, coff, _so, phys) in self.g.rank_chunks(r):
                    if rows:
                        a = self.units[u][5] + coff
                        fill_device(sh[phys:phys + rows * cols], ps, self.units, a, a + rows * cols)
                if r in self.g.state:
                    m0 = self.g.state[r]["master"][0]
                    for c in self.g.rank_chunks(r):
                        phys, n = c[9], c[6] * c[5]
                        m0[phys:phys + n] = sh[phys:phys + n].view(t16).float()
        else:
            ranks = list(range(w.n_d)) if peers else self.bound
            for r in ranks:
                sh = self.g.shard16[r] if r in self.g.shard16 else self.g.bind_peer_shard(r)
                for (u, off, n, base, S) in self.g.shard_slices(r):
                    if n:
                        fill_device(sh[off:off + n], ps, self.units, base + r * S, base + (r + 1) * S)
                if r in self.g.state:
                    m0 = self.g.state[r]["master"][0]
                    for (u, off, n, base, S) in self.g.shard_slices(r):
                        m0[off:off + n] = sh[off:off + n].view(t16).float()
        self.scaler = None
        if w.scaler is not None:
            c = w.scaler
            self.scaler = Z.scaler(c.init_scale, c.growth_factor, c.backoff_factor, c.min_scale,
                                   c.growth_interval)
            self.g.set_scaler(self.scaler)
        self.hyper = Z.hyper(w.hyper.lr, w.hyper.beta1, w.hyper.beta2, w.hyper.eps,
                             w.hyper.weight_decay, w.hyper.max_grad_norm, w.hyper.report_norm)
        n_c = int(self.info.max_contrib_elems) if alloc_contribs else 0
        self.contribs = [torch.empty(max(8, n_c), dtype=torch.int16, device="cuda")
                         for _ in range(w.n_d)]
        self.gather_buf = None
        if w.stage == 3:
            self.gather_buf = torch.empty(max(8, int(self.info.max_unit_pad)), dtype=torch.int16,
                                          device="cuda")

    def ranges(self):
        """(which, lo, hi) of each zero_step call of a step."""
        if self.w.stage == 3:
            return [(u, U[5], U[5] + U[3]) for u, U in enumerate(self.units)]
        B = self.w.bucket_elems or int(self.info.phi_pad)
        return [(b, b * B, min((b + 1) * B, int(self.info.phi_pad)))
                for b in range(int(self.info.n_buckets))]

    def step(self, k: int, gather_check=None):
        """Run 1-based step k: (stage 3: gather, then) reduce + update per bucket / unit.
        With clipping, a gradient-norm pass over every bucket / unit comes first."""
        if self.w.hyper.max_grad_norm > 0:
            for which, lo, hi in self.ranges():
                for r in range(self.w.n_d):
                    fill_device(self.contribs[r], grad_stream(self.w, k, r), self.units, lo, hi)
                self.g.grad_norm([c.data_ptr() for c in self.contribs], which)
        for which, lo, hi in self.ranges():
            if self.w.stage == 3:
                self.g.gather(which, self.gather_buf)
                if gather_check is not None:
                    gather_check(which, lo, hi, self.gather_buf)
                self.g.release(which)
            for r in range(self.w.n_d):
                fill_device(self.contribs[r], grad_stream(self.w, k, r), self.units, lo, hi)
            self.g.step([c.data_ptr() for c in self.contribs], which, self.hyper)
        return self.g.finish()

    # ------------------------------------------------------------------ readback
    def locate(self, idx: np.ndarray):
        """(rank, physical offset) of flat indices; rank -1 when not owned by a bound rank."""
        rank = np.full(idx.size, -1, dtype=np.int64)
        phys = np.zeros(idx.size, dtype=np.int64)
        if self.w.per_param:
            ch = np.array([c for c in self.g.chunks if c[4] > 0], dtype=np.int64).reshape(-1, 10)
            start = np.array([self.units[int(u)][5] for u in ch[:, 1]], dtype=np.int64) + ch[:, 7]
            order = np.argsort(start)
            start, ch = start[order], ch[order]
            j = np.searchsorted(start, idx, side="right") - 1
            ok = (j >= 0)
            j = np.clip(j, 0, max(0, len(start) - 1))
            ok &= idx < start[j] + ch[j, 4] * ch[j, 5]
            rank[ok] = ch[j[ok], 0]
            phys[ok] = ch[j[ok], 9] + idx[ok] - start[j[ok]]
            rank[~np.isin(rank, self.bound)] = -1
            return rank, phys
        for u, (_f, _c, _n, numel_pad, S, base, _sb) in enumerate(self.units):
            sel = (idx >= base) & (idx < base + numel_pad)
            if not sel.any() or S == 0:
                continue
            loc = idx[sel] - base
            r = loc // S
            ph = np.zeros(loc.size, dtype=np.int64)
            for rr in np.unique(r):
                mk = r == rr
                ph[mk] = self.g.phys_off[int(rr)][u] + loc[mk] - rr * S
            rank[sel] = r
            phys[sel] = ph
        rank[~np.isin(rank, self.bound)] = -1
        return rank, phys

    def read_sampled(self, idx: np.ndarray):
        rank, phys = self.locate(idx)
        assert (rank >= 0).all()
        out = {k: np.zeros(idx.size, np.float32) for k in ("master", "m", "v")}
        out16 = np.zeros(idx.size, np.uint16)
        for r in np.unique(rank):
            sel = np.nonzero(rank == r)[0]
            pi = torch.from_numpy(phys[sel]).cuda()
            for k in out:
                t = self.g.state_tensor(int(r), k)
                out[k][sel] = t[pi.to(t.device)].cpu().numpy()
            if self.w.stage == 3:
                out16[sel] = self.g.shard16[int(r)][pi].cpu().numpy().view(np.uint16)
        if self.w.stage != 3:
            out16 = self.g.full16[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint16)
        return out, out16

    def read_logical(self, r: int):
        return {k: self.g.logical(r, self.g.state_tensor(r, k)).cpu().numpy()
                for k in ("master", "m", "v")}

    def close(self):
        self.g.close()
        del self.contribs
        torch.cuda.empty_cache()
