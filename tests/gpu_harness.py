"""GPU-side harness for parity tests: seeded inputs on the device, oracle replay on the host.

The device inputs come from the shared generator (synth); the expected values come only
from the oracle, run on host copies of the same seeded streams.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import zero_sharded_mixed_03_gb300 as Z
from synth import workloads as W
from zero_sharded_mixed_03_gb300.emulate import EmulatedGroup

TORCH16 = {W.BF16: torch.bfloat16, W.FP16: torch.float16}


def _unit_parts(units, lo, hi):
    """Split [lo, hi) of the global flat space into (a, e, real) pieces (real = inside a tensor)."""
    out = []
    for (_f, _c, numel, numel_pad, _s, base, _sb) in units:
        for a, e, real in ((base, base + numel, True), (base + numel, base + numel_pad, False)):
            a2, e2 = max(a, lo), min(e, hi)
            if a2 < e2:
                out.append((a2, e2, real))
    return out


def fill_device(dst: torch.Tensor, stream: synth.Stream, units, lo: int, hi: int) -> None:
    """dst[j] = stream value at flat index lo + j, zero in padding."""
    assert dst.numel() >= hi - lo and dst.dtype == torch.int16
    cs = torch.cuda.current_stream().cuda_stream
    for a, e, real in _unit_parts(units, lo, hi):
        if real:
            stream.device(dst.data_ptr() + 2 * (a - lo), a, e - a, cs)
        else:
            dst[a - lo:e - lo].zero_()


def fill_host(stream: synth.Stream, units, lo: int, hi: int) -> np.ndarray:
    out = np.zeros(hi - lo, dtype=np.uint16)
    for a, e, real in _unit_parts(units, lo, hi):
        if real:
            stream.host_into(out[a - lo:e - lo], a)
    return out


def values_at(stream: synth.Stream, units, idx: np.ndarray) -> np.ndarray:
    """Stream values at flat indices idx (zero at padding)."""
    out = stream.at(idx)
    real = np.zeros(idx.size, dtype=bool)
    for (_f, _c, numel, _np, _s, base, _sb) in units:
        real |= (idx >= base) & (idx < base + numel)
    out[~real] = 0
    return out


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
        ps = synth.param_stream(w)
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
                    fill_device(self.contribs[r], synth.grad_stream(self.w, k, r), self.units, lo, hi)
                self.g.grad_norm([c.data_ptr() for c in self.contribs], which)
        for which, lo, hi in self.ranges():
            if self.w.stage == 3:
                self.g.gather(which, self.gather_buf)
                if gather_check is not None:
                    gather_check(which, lo, hi, self.gather_buf)
                self.g.release(which)
            for r in range(self.w.n_d):
                fill_device(self.contribs[r], synth.grad_stream(self.w, k, r), self.units, lo, hi)
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


# ---------------------------------------------------------------------- oracle side

def expected_flag(w: W.Workload, k: int) -> int:
    """Non-finite flag of step k.  Generated contributions are bounded (|value| <= 3.47
    sigma, x100 for outliers), so sums of N_d of them are finite: only a planted inf flags."""
    return int(w.inject is not None and w.inject[0] == k)


def oracle_units(w: W.Workload):
    """(first, count, numel, numel_pad, shard, base, shard_base) of every unit, from the
    oracle's own partition (per-parameter plans: unpadded unit buffers)."""
    if w.per_param:
        pp = oracle.PerParam(w.sizes, w.dim0, w.n_d, w.unit_first or None)
        return [(0, 0, n, n, 0, int(b), 0) for n, b in zip(pp.unit_numel, pp.unit_base[:-1])]
    L = oracle.Layout(w.sizes, w.n_d, w.unit_first or None)
    return [tuple(int(x) for x in u) for u in L.units]


class OracleSampled:
    """Oracle trajectory of the sampled flat indices (elementwise replay of every step)."""

    def __init__(self, w: W.Workload, idx: np.ndarray):
        self.w, self.idx = w, idx
        units = oracle_units(w)
        self.units = units
        p16 = values_at(synth.param_stream(w), units, idx)
        self.p = oracle.widen16(p16, w.dtype).astype(np.float32)
        self.m = np.zeros(idx.size, np.float32)
        self.v = np.zeros(idx.size, np.float32)
        self.out16 = p16.copy()
        self.sc = oracle.ScalerState(w.scaler)

    def step(self, k: int) -> int:
        w = self.w
        c = [values_at(synth.grad_stream(w, k, r), self.units, self.idx) for r in range(w.n_d)]
        k9 = oracle.consts(w.hyper, self.sc.t + 1, self.sc.scale, w.n_d)
        g, seen = oracle.reduce(c, w.dtype, float(k9[8]))
        flag = expected_flag(w, k)
        assert seen <= flag
        if flag:
            oracle.recast(self.p, w.dtype, self.out16)
        else:
            oracle.adamw(g, self.p, self.m, self.v, k9, w.dtype, self.out16)
        self.sc.update(flag)
        return flag


class OracleFull:
    """Oracle over whole host buffers (small workloads)."""

    def __init__(self, w: W.Workload, bound):
        self.w = w
        self.units = oracle_units(w)
        self.bound = [1 if r in bound else 0 for r in range(w.n_d)]
        self.p, self.m, self.v, self.sh16 = [], [], [], []
        self.sc = oracle.ScalerState(w.scaler)
        if w.per_param:
            assert w.hyper.max_grad_norm == 0
            self.pp = oracle.PerParam(w.sizes, w.dim0, w.n_d, w.unit_first or None)
            self.total = int(self.pp.unit_base[-1])
            self.params16 = fill_host(synth.param_stream(w), self.units, 0, self.total)
            for r in range(w.n_d):
                P = np.zeros(max(1, self.pp.per_rank), np.float32)
                S16 = np.zeros(max(1, self.pp.per_rank), np.uint16)
                for (rr, u, t, row0, rows, cols, c_rows, coff, soff) in self.pp.chunks:
                    if rr == r and rows:
                        g0 = self.pp.unit_base[u] + coff
                        S16[soff:soff + rows * cols] = self.params16[g0:g0 + rows * cols]
                P[:] = oracle.widen16(S16, w.dtype)
                self.p.append(P)
                self.m.append(np.zeros_like(P))
                self.v.append(np.zeros_like(P))
                self.sh16.append(S16)
            return
        self.L = oracle.Layout(w.sizes, w.n_d, w.unit_first or None)
        n = self.L.total_pad
        self.params16 = fill_host(synth.param_stream(w), self.units, 0, n)
        for r in range(w.n_d):
            idx = np.concatenate([np.arange(U[5] + r * U[4], U[5] + (r + 1) * U[4]) for U in self.units]) \
                if self.units else np.zeros(0, np.int64)
            idx = idx.astype(np.int64)
            self.p.append(oracle.widen16(self.params16[idx], w.dtype).astype(np.float32))
            self.m.append(np.zeros(idx.size, np.float32))
            self.v.append(np.zeros(idx.size, np.float32))
            self.sh16.append(self.params16[idx].copy())
        self.full16 = self.params16.copy()

    def step(self, k: int) -> int:
        w = self.w
        if w.per_param:
            c = [fill_host(synth.grad_stream(w, k, r), self.units, 0, self.total) for r in range(w.n_d)]
            k9 = oracle.consts(w.hyper, self.sc.t + 1, self.sc.scale, w.n_d)
            flag = self.pp.step(w.dtype, c, self.bound, self.p, self.m, self.v, self.sh16, k9)
            self.norm2 = float("nan")
            self.sc.update(flag)
            return flag
        n = self.L.total_pad
        c = [fill_host(synth.grad_stream(w, k, r), self.units, 0, n) for r in range(w.n_d)]
        k9 = oracle.consts(w.hyper, self.sc.t + 1, self.sc.scale, w.n_d)
        flag, self.norm2 = oracle.sharded_step_ex(
            self.L, w.stage, w.bucket_elems, w.dtype, c, self.bound, self.p, self.m, self.v,
            self.sh16 if w.stage == 3 else None, self.full16 if w.stage != 3 else None, k9,
            w.hyper.max_grad_norm)
        self.sc.update(flag)
        return flag

    def gathered(self, u: int) -> np.ndarray:
        if self.w.per_param:
            return self.pp.gather(u, self.sh16)
        return oracle.gather_unit(self.L, u, self.sh16)


# ---------------------------------------------------------------------- comparisons

def ordered16(h: np.ndarray) -> np.ndarray:
    """Map 16-bit float patterns to integers ordered like their values (+0 == -0)."""
    h = h.astype(np.int64)
    mag = h & 0x7FFF
    return np.where(h & 0x8000, -mag, mag)


def assert_state_close(got: np.ndarray, want: np.ndarray, what: str):
    """fp32 tolerance: |got - want| <= 1e-6 |want| + 1e-8 (and report bit mismatches)."""
    diff = np.abs(got.astype(np.float64) - want.astype(np.float64))
    tol = 1e-6 * np.abs(want.astype(np.float64)) + 1e-8
    bad = np.nonzero(~(diff <= tol))[0]
    assert bad.size == 0, f"{what}: {bad.size} elements out of tolerance, first at {bad[0]}: " \
                          f"got {got[bad[0]]!r} want {want[bad[0]]!r}"
    return int(np.count_nonzero(got.view(np.uint32) != want.view(np.uint32)))


def assert_16_close(got: np.ndarray, want: np.ndarray, what: str):
    """16-bit tolerance: at most one unit in the last place."""
    d = np.abs(ordered16(got) - ordered16(want))
    bad = np.nonzero(d > 1)[0]
    assert bad.size == 0, f"{what}: {bad.size} elements beyond 1 ulp, first at {bad[0]}: " \
                          f"got {got[bad[0]]:#06x} want {want[bad[0]]:#06x}"
    return int(np.count_nonzero(got != want))


def sample_indices(run: Run, n_random: int = 20000, seed: int = 0,
                   bound_only: bool = True) -> np.ndarray:
    """Random flat indices plus every boundary the kernel treats specially: shard, bucket,
    unit, tensor and padding edges (each +-9 elements), restricted to bound ranks."""
    rng = np.random.default_rng(seed)
    n = int(run.info.phi_pad)
    pts = [rng.integers(0, max(1, n), size=n_random)]
    edges = [0, n]
    for (_f, _c, numel, numel_pad, S, base, _sb) in run.units:
        edges += [base, base + numel, base + numel_pad]
        edges += [base + r * S for r in range(run.w.n_d + 1)]
    if run.w.stage != 3 and run.w.bucket_elems:
        edges += list(range(0, n, run.w.bucket_elems))
    if run.w.per_param:                               # every rank's row-chunk boundaries
        edges += [run.units[c[1]][5] + c[7] for c in run.g.chunks]
    if run.w.per_param:
        offs = np.concatenate([[0], np.cumsum(run.w.sizes)[:-1]]).astype(np.int64)
    else:
        offs = oracle.Layout(run.w.sizes, run.w.n_d, run.w.unit_first or None).tensor_offset
    pick = offs[rng.integers(0, offs.size, size=min(400, offs.size))] if offs.size else []
    edges += [int(x) for x in pick]
    e = np.array(edges, dtype=np.int64)
    pts.append((e[:, None] + np.arange(-9, 10)[None, :]).ravel())
    idx = np.unique(np.concatenate(pts))
    idx = idx[(idx >= 0) & (idx < n)]
    if not bound_only:
        return idx
    rank, _ = run.locate(idx)
    return idx[rank >= 0]
