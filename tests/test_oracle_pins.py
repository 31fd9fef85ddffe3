"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against a value the pages print, a closed form, an
invariant, a library routine (numpy / torch) or brute force on tiny inputs.
"""
import fractions
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BF16, FP16 = 0, 1


def _golden_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                out[k] = v
    return out


# ----------------------------------------------------------------- 16-bit encodings

def _float_patterns(n, seed=0):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    # bias towards the exponent range of the 16-bit formats, including subnormals/overflow
    e = rng.integers(90, 150, size=n // 2).astype(np.uint32)
    bits[: n // 2] = (bits[: n // 2] & 0x807FFFFF) | (e << 23)
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x00000001,
                        0x477FEFFF, 0x477FF000, 0x477FF001, 0x33000000, 0x33000001, 0x32FFFFFF,
                        0x387FC000, 0x387FE000, 0x38800000, 0x3F808000, 0x3F818000, 0x3F80C000,
                        0x7F7F8000, 0x7F7F7FFF], dtype=np.uint32)
    # every fp16 value and its neighbours at +- half an fp16 ulp (ties)
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    hv = h.view(np.float16).astype(np.float32).view(np.uint32)
    ties = np.concatenate([hv, hv + 1, hv - 1, (hv + 0x1000), hv + 0xFFF])
    return np.concatenate([bits, special, ties]).view(np.float32)


@pytest.mark.parametrize("is_fp16", [0, 1])
def test_round16_matches_library(is_fp16):
    f = _float_patterns(400_000)
    f = f[~np.isnan(f)]
    got = oracle.round16(f, is_fp16)
    if is_fp16:
        want = f.astype(np.float16).view(np.uint16)       # numpy: IEEE round-to-nearest-even
    else:
        want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (hex(f.view(np.uint32)[bad[0]]), hex(got[bad[0]]), hex(want[bad[0]]))


@pytest.mark.parametrize("is_fp16", [0, 1])
def test_round16_nan_stays_nan(is_fp16):
    got = oracle.round16(np.array([np.nan, -np.nan], dtype=np.float32), is_fp16)
    exp_mask = 0x7C00 if is_fp16 else 0x7F80
    man_mask = 0x03FF if is_fp16 else 0x007F
    assert all((g & exp_mask) == exp_mask and (g & man_mask) != 0 for g in got)


@pytest.mark.parametrize("is_fp16", [0, 1])
def test_widen16_all_patterns(is_fp16):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen16(h, is_fp16)
    if is_fp16:
        want = h.view(np.float16).astype(np.float32)
    else:
        want = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


@pytest.mark.parametrize("is_fp16", [0, 1])
def test_generator_rounding_matches_library(is_fp16):
    lib = synth._load_host()
    f = _float_patterns(20_000, seed=3)
    f = f[~np.isnan(f)]
    fn = lib.syn_round_fp16 if is_fp16 else lib.syn_round_bf16
    got = np.array([fn(float(x)) for x in f], dtype=np.uint16)
    if is_fp16:
        want = f.astype(np.float16).view(np.uint16)
    else:
        want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


# ----------------------------------------------------------------- memory accounting

def test_memory_closed_forms_table():
    g = _golden_kv("closed_forms.txt")
    rng = np.random.default_rng(1)
    for _ in range(200):
        n_d = int(rng.integers(1, 130))
        phi = int(rng.integers(0, 10**9)) * n_d       # divisible: the pages' forms hold exactly
        mem = oracle.memory(phi, n_d)
        for s, name in enumerate(["ddp", "zero1", "zero2", "zero3"]):
            vals = g[name]
            for j in range(3):
                num, den = int(vals[2 * j]), vals[2 * j + 1]
                den = n_d if den == "N" else int(den)
                assert mem[3 * s + j] * den == num * phi, (name, j)
        # totals as printed: 16Phi, 4Phi + 12Phi/N, 2Phi + 14Phi/N, 16Phi/N
        assert mem[0:3].sum() == int(g["bytes_per_param"][0]) * phi
        assert mem[3:6].sum() * n_d == 4 * phi * n_d + 12 * phi
        assert mem[6:9].sum() * n_d == 2 * phi * n_d + 14 * phi
        assert mem[9:12].sum() * n_d == 16 * phi
        assert mem[12] == int(g["fp32_grad_ddp_total"][0]) * phi


def test_memory_worked_example_70b():
    g = _golden_kv("memory_70b_nd64.txt")
    phi, n_d = int(g["phi"][0]), int(g["n_d"][0])
    mem = oracle.memory(phi, n_d)
    totals = [mem[3 * s:3 * s + 3].sum() / 1e9 for s in range(4)]
    for got, key in zip(totals, ["ddp_gb", "zero1_gb", "zero2_gb", "zero3_gb"]):
        assert round(got, 1) == float(g[key][0]), key
    m5 = oracle.memory(int(g["phi_5b"][0]), 1)
    assert m5[0:3].sum() / 1e9 == float(g["ddp_5b_gb"][0])


def test_memory_limits_4x_8x():
    g = _golden_kv("closed_forms.txt")
    phi = 10**6
    prev1 = prev2 = 0.0
    for n_d in [1, 2, 8, 64, 1000, 10**6]:
        mem = oracle.memory(phi * n_d, n_d)
        r1 = mem[0:3].sum() / mem[3:6].sum()
        r2 = mem[0:3].sum() / mem[6:9].sum()
        assert prev1 <= r1 <= float(g["limit_zero1"][0]) and prev2 <= r2 <= float(g["limit_zero2"][0])
        prev1, prev2 = r1, r2
    assert abs(prev1 - 4.0) < 1e-4 and abs(prev2 - 8.0) < 1e-4


# ----------------------------------------------------------------- communication

def test_comm_closed_forms():
    g = _golden_kv("closed_forms.txt")
    rng = np.random.default_rng(2)
    for _ in range(300):
        n_d = int(rng.integers(1, 200))
        phi = int(rng.integers(0, 10**9)) * n_d
        c = oracle.comm(phi, n_d)
        one = (n_d - 1) * phi // n_d                 # (N-1)/N * Phi, one ring collective
        assert (n_d - 1) * phi % n_d == 0
        assert c[0] == int(g["comm_ddp"][0]) * one
        assert c[1] == c[2] == int(g["comm_zero12"][0]) * one == c[0]   # no overhead over DDP
        assert c[3] == int(g["comm_zero3"][0]) * one
        if c[0]:
            assert fractions.Fraction(int(c[3]), int(c[0])) == fractions.Fraction(g["comm_ratio"][0])
    assert list(oracle.comm(1000, 1)) == [0, 0, 0, 0]


# ----------------------------------------------------------------- tables, brute force

def _brute_layout(sizes, n_d, unit_first):
    firsts = list(unit_first) if unit_first else [0]
    ends = firsts[1:] + [len(sizes)]
    units, base, sbase, toff = [], 0, 0, [0] * len(sizes)
    for f, e in zip(firsts, ends):
        numel = 0
        for t in range(f, e):
            toff[t] = base + numel
            numel += sizes[t]
        pad = numel
        while pad % n_d:
            pad += 1
        units.append((f, e - f, numel, pad, pad // n_d, base, sbase))
        base += pad
        sbase += pad // n_d
    return units, toff


def _brute_segments(sizes, n_d, unit_first):
    """Walk every element of every shard; owner tensor by linear search."""
    units, toff = _brute_layout(sizes, n_d, unit_first)
    rows = []
    for r in range(n_d):
        for u, (f, cnt, numel, pad, S, base, sbase) in enumerate(units):
            cur = None
            for i in range(S):
                gidx = base + r * S + i
                owner = -1
                for t in range(f, f + cnt):
                    if toff[t] <= gidx < toff[t] + sizes[t]:
                        owner = t
                if cur is not None and cur[2] == owner:
                    cur[5] += 1
                else:
                    if cur is not None:
                        rows.append(cur)
                    in_off = gidx - toff[owner] if owner >= 0 else gidx - (base + numel)
                    cur = [r, u, owner, in_off, sbase + i, 1]
            if cur is not None:
                rows.append(cur)
    return units, toff, rows


def _random_case(rng, max_tensors=12, max_size=9, units=True):
    nt = int(rng.integers(0, max_tensors + 1))
    sizes = [int(x) for x in rng.integers(0, max_size + 1, size=nt)]
    unit_first = []
    if units and nt > 0 and rng.random() < 0.6:
        cuts = sorted(set(int(x) for x in rng.integers(1, nt + 1, size=int(rng.integers(0, 4)))) - {nt})
        unit_first = [0] + [c for c in cuts if 0 < c < nt]
    return sizes, unit_first


def test_tables_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(400):
        sizes, unit_first = _random_case(rng)
        n_d = int(rng.integers(1, 10))
        L = oracle.Layout(sizes, n_d, unit_first)
        units, toff, rows = _brute_segments(sizes, n_d, unit_first)
        assert [tuple(int(x) for x in u) for u in L.units] == units
        assert list(L.tensor_offset) == toff
        assert [list(map(int, r)) for r in L.shard_segments()] == rows
        for u in units:   # pad to the smallest multiple of N_d
            assert u[3] % n_d == 0 and 0 <= u[3] - u[2] < n_d


def test_bucket_segments_brute_force():
    rng = np.random.default_rng(4)
    for _ in range(300):
        n_d = int(rng.integers(1, 10))
        phi_pad = int(rng.integers(0, 60)) * n_d
        B = int(rng.integers(0, 25))
        L = oracle.lib()
        n = L.orc_bucket_segments(phi_pad, n_d, B, None, 0)
        rows = np.zeros((max(1, n), 5), dtype=np.int64)
        L.orc_bucket_segments(phi_pad, n_d, B, rows.ctypes.data, n)
        rows = rows[:n]
        # brute force: label every element with (bucket, rank) and cut runs
        S = phi_pad // n_d
        BB = B if B else max(phi_pad, 1)
        want = []
        for b in range((phi_pad + BB - 1) // BB if phi_pad else 0):
            for r in range(n_d):
                idx = [i for i in range(b * BB, min((b + 1) * BB, phi_pad)) if i // S == r] if S else []
                if idx:
                    want.append([b, r, idx[0], idx[0] - r * S, len(idx)])
        assert [list(map(int, x)) for x in rows] == want


# ----------------------------------------------------------------- step semantics

def _rand16(rng, shape, is_fp16, scale=0.01):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return oracle.round16(x, is_fp16)


def _zero_pad(arr, L):
    for U in L.units:
        arr[int(U[5] + U[2]):int(U[5] + U[3])] = 0
    return arr


def _run_sharded(L, stage, bucket, is_fp16, contribs, params16, k9, bound=None):
    n_d = L.n_d
    bound = bound if bound is not None else [1] * n_d
    p, m, v, sh16 = [], [], [], []
    for r in range(n_d):
        idx = np.concatenate([np.arange(U[5] + r * U[4], U[5] + (r + 1) * U[4]) for U in L.units]) \
            if len(L.units) else np.zeros(0, dtype=np.int64)
        idx = idx.astype(np.int64)
        p.append(oracle.widen16(params16[idx], is_fp16).astype(np.float32))
        m.append(np.zeros(idx.size, dtype=np.float32))
        v.append(np.zeros(idx.size, dtype=np.float32))
        sh16.append(params16[idx].copy())
    full = params16.copy()
    flag = oracle.sharded_step(L, stage, bucket, is_fp16, contribs, bound, p, m, v,
                               sh16 if stage == 3 else None, full if stage != 3 else None, k9)
    return flag, p, m, v, sh16, full


def _union(L, parts):
    out = np.zeros(L.total_pad, dtype=parts[0].dtype)
    for r, a in enumerate(parts):
        for U in L.units:
            out[U[5] + r * U[4]:U[5] + (r + 1) * U[4]] = a[U[6]:U[6] + U[4]]
    return out


def test_sharded_equals_ddp_bit_exact():
    """[ZF] 'Mathematical Formulation of ZeRO Partitioning Stages': partitioning keeps the
    exact semantics of standard data parallelism -> union of shard updates == DDP step."""
    rng = np.random.default_rng(5)
    hyper = W.Hyper()
    for trial in range(300):
        sizes, unit_first = _random_case(rng, max_tensors=10, max_size=9)
        n_d = int(rng.integers(1, 10))
        stage = int(rng.integers(1, 4))
        if stage != 3:
            unit_first = []
        is_fp16 = int(rng.integers(0, 2))
        L = oracle.Layout(sizes, n_d, unit_first)
        n = L.total_pad
        bucket = int(rng.integers(0, 12)) if stage != 3 else 0
        params16 = _zero_pad(_rand16(rng, n, is_fp16, 0.02), L)
        contribs = [_zero_pad(_rand16(rng, n, is_fp16), L) for _ in range(n_d)]
        t = int(rng.integers(1, 6))
        scale = float(2.0 ** int(rng.integers(0, 17))) if is_fp16 else 1.0
        k9 = oracle.consts(hyper, t, scale, n_d)
        flag, p, m, v, sh16, full = _run_sharded(L, stage, bucket, is_fp16, contribs, params16, k9)
        P = oracle.widen16(params16, is_fp16).astype(np.float32)
        M = np.zeros(n, np.float32)
        V = np.zeros(n, np.float32)
        out = np.zeros(n, np.uint16)
        f2 = oracle.ddp_step(contribs, is_fp16, P, M, V, out, k9)
        assert flag == f2 == 0
        assert np.array_equal(_union(L, p).view(np.uint32), P.view(np.uint32)), trial
        assert np.array_equal(_union(L, m).view(np.uint32), M.view(np.uint32))
        assert np.array_equal(_union(L, v).view(np.uint32), V.view(np.uint32))
        got16 = _union(L, sh16) if stage == 3 else full
        assert np.array_equal(got16, out)


def test_bucketing_invariance():
    rng = np.random.default_rng(6)
    hyper = W.Hyper()
    for _ in range(60):
        sizes, _ = _random_case(rng, max_tensors=12, max_size=20, units=False)
        n_d = int(rng.integers(1, 9))
        L = oracle.Layout(sizes, n_d)
        n = L.total_pad
        params16 = _zero_pad(_rand16(rng, n, 0, 0.02), L)
        contribs = [_zero_pad(_rand16(rng, n, 0), L) for _ in range(n_d)]
        k9 = oracle.consts(hyper, 1, 1.0, n_d)
        ref = _run_sharded(L, 2, 0, 0, contribs, params16, k9)
        for B in [1, 3, 7, 16, n + 5]:
            got = _run_sharded(L, 2, B, 0, contribs, params16, k9)
            for a, b in zip(ref[1] + ref[2] + ref[3], got[1] + got[2] + got[3]):
                assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
            assert np.array_equal(ref[5], got[5])


def test_padding_stays_zero():
    hyper = W.Hyper()
    rng = np.random.default_rng(7)
    sizes = [5, 3, 1]          # phi 9, N 4 -> pad 3
    L = oracle.Layout(sizes, 4)
    n = L.total_pad
    assert n == 12
    params16 = _zero_pad(_rand16(rng, n, 0, 0.02), L)
    full = params16.copy()
    p = [oracle.widen16(params16[r * 3:(r + 1) * 3], 0).astype(np.float32) for r in range(4)]
    m = [np.zeros(3, np.float32) for _ in range(4)]
    v = [np.zeros(3, np.float32) for _ in range(4)]
    for t in range(1, 6):
        contribs = [_zero_pad(_rand16(rng, n, 0), L) for _ in range(4)]
        k9 = oracle.consts(hyper, t, 1.0, 4)
        assert oracle.sharded_step(L, 1, 0, 0, contribs, [1] * 4, p, m, v, None, full, k9) == 0
    assert np.all(full[9:] == 0)
    assert np.all(p[3] == 0) and np.all(m[3] == 0) and np.all(v[3] == 0)


@pytest.mark.parametrize("bits", [0x7F80, 0xFF80, 0x7FC1])
def test_skip_on_nonfinite_keeps_state(bits):
    hyper = W.Hyper()
    rng = np.random.default_rng(8)
    L = oracle.Layout([17, 30], 3)
    n = L.total_pad
    params16 = _zero_pad(_rand16(rng, n, 0, 0.02), L)
    contribs = [_zero_pad(_rand16(rng, n, 0), L) for _ in range(3)]
    contribs[2][23] = bits
    k9 = oracle.consts(hyper, 1, 1.0, 3)
    flag, p, m, v, _, full = _run_sharded(L, 2, 7, 0, contribs, params16, k9)
    assert flag == 1
    p0 = [oracle.widen16(params16[r * 16:(r + 1) * 16], 0) for r in range(3)]
    for r in range(3):
        assert np.array_equal(p[r].view(np.uint32), p0[r].view(np.uint32))
        assert not m[r].any() and not v[r].any()
    assert np.array_equal(full, params16)   # re-cast of the unchanged master


def test_overflowing_finite_sum_is_flagged():
    # bf16 has fp32's exponent range: two finite 3e38 contributions overflow the fp32 sum
    big = oracle.round16(np.array([3.0e38], np.float32), 0)
    g, flag = oracle.reduce([big, big], 0, 0.5)
    assert flag == 1 and np.isinf(g[0])
    g, flag = oracle.reduce([big, oracle.round16(np.array([-3.0e38], np.float32), 0)], 0, 0.5)
    assert flag == 0 and g[0] == 0.0


def test_reduce_exact_sums():
    """Contributions that are small multiples of 2^-10 sum exactly in fp32; with
    N * scale a power of two the scaled result is exact: compare with rationals."""
    rng = np.random.default_rng(9)
    for n_d in [1, 2, 3, 4, 7, 8, 16]:
        for is_fp16, scale in [(0, 1.0), (1, 1024.0)]:
            ints = rng.integers(-255, 256, size=(n_d, 64))
            vals = (ints / 1024.0).astype(np.float32)
            c = [oracle.round16(vals[r], is_fp16) for r in range(n_d)]
            assert all(np.array_equal(oracle.widen16(c[r], is_fp16), vals[r]) for r in range(n_d))
            inv = np.float32(1.0 / (n_d * scale))
            g, flag = oracle.reduce(c, is_fp16, inv)
            assert flag == 0
            for i in range(64):
                exact = sum(fractions.Fraction(int(ints[r, i]), 1024) for r in range(n_d))
                want = exact * fractions.Fraction(float(inv))
                if (n_d & (n_d - 1)) == 0:
                    assert fractions.Fraction(float(g[i])) == want
                else:   # one rounding of the exact product
                    assert abs(fractions.Fraction(float(g[i])) - want) <= abs(want) * fractions.Fraction(1, 2**23)


def test_average_and_unscale_invariant():
    """[ZF] 'Execution Flow for ZeRO-1': each rank receives the AVERAGED gradient of its
    partition.  N identical contributions, each multiplied by the loss scale (a power of
    two, exact), must give the same update as one unscaled contribution: the step
    averages over N_d and divides out the loss scale."""
    hyper = W.Hyper()
    rng = np.random.default_rng(14)
    sizes = [37, 11, 64]
    for is_fp16, scale in [(0, 1.0), (1, 1.0), (1, 1024.0), (0, 65536.0)]:
        base = _rand16(rng, 112, is_fp16)
        params16 = _rand16(rng, 112, is_fp16, 0.02)
        L1 = oracle.Layout(sizes, 1)
        ref = _run_sharded(L1, 1, 0, is_fp16, [base], params16, oracle.consts(hyper, 2, 1.0, 1))
        scaled = oracle.round16(oracle.widen16(base, is_fp16) * np.float32(scale), is_fp16)
        assert np.array_equal(oracle.widen16(scaled, is_fp16),
                              oracle.widen16(base, is_fp16) * np.float32(scale))
        for n_d in [2, 4, 8, 16]:
            L = oracle.Layout(sizes, n_d)
            k9 = oracle.consts(hyper, 2, scale, n_d)
            got = _run_sharded(L, 1, 0, is_fp16, [scaled] * n_d, params16, k9)
            assert np.array_equal(_union(L, got[1]).view(np.uint32), ref[1][0].view(np.uint32))
            assert np.array_equal(got[5], ref[5])


def test_adamw_matches_torch_optim():
    """N_d = 1, loss scale 1: the step is plain mixed-precision AdamW on the widened
    gradient; cross-check the fp32 master/m/v against torch.optim.AdamW (CPU, fp32)."""
    hyper = W.Hyper()
    rng = np.random.default_rng(10)
    n = 4096
    p0 = oracle.widen16(_rand16(rng, n, 0, 0.02), 0).astype(np.float32)
    P, M, V = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=hyper.lr, betas=(hyper.beta1, hyper.beta2), eps=hyper.eps,
                            weight_decay=hyper.weight_decay, foreach=False)
    for t in range(1, 8):
        c = _rand16(rng, n, 0, 0.01)
        g = oracle.widen16(c, 0).astype(np.float32)
        k9 = oracle.consts(hyper, t, 1.0, 1)
        oracle.adamw(g, P, M, V, k9, 0)
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
        st = opt.state[tp]
        for mine, ref in [(P, tp.detach().numpy()), (M, st["exp_avg"].numpy()),
                          (V, st["exp_avg_sq"].numpy())]:
            assert np.all(np.abs(mine - ref) <= 1e-6 * np.abs(ref) + 1e-8), t


def test_adamw_first_step_closed_forms():
    """t = 1 from m = v = 0: m = (1-b1) g, v = (1-b2) g^2 and, since sqrt(v)/sqrt(1-b2) = |g|,
    the update is p(1 - lr wd) - lr g / (|g| + eps)."""
    hyper = W.Hyper()
    rng = np.random.default_rng(11)
    n = 2000
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    P, M, V = p.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    k9 = oracle.consts(hyper, 1, 1.0, 1)
    oracle.adamw(g, P, M, V, k9, 0)
    assert np.array_equal(M, np.float32(1 - hyper.beta1) * g)
    assert np.array_equal(V, np.float32(1 - hyper.beta2) * (g * g))
    pd, gd = p.astype(np.float64), g.astype(np.float64)
    want = pd * (1 - hyper.lr * hyper.weight_decay) - hyper.lr * gd / (np.abs(gd) + hyper.eps)
    assert np.all(np.abs(P - want) <= 2e-7 * np.abs(want) + 1e-9)


def test_zero_gradient_is_pure_decay():
    hyper = W.Hyper()
    p = (np.random.default_rng(12).standard_normal(500) * 0.02).astype(np.float32)
    P, M, V = p.copy(), np.zeros(500, np.float32), np.zeros(500, np.float32)
    for t in range(1, 4):
        oracle.adamw(np.zeros(500, np.float32), P, M, V, oracle.consts(hyper, t, 1.0, 1), 0)
        p = p - np.float32(hyper.lr * hyper.weight_decay) * p
        assert np.array_equal(P, p) and not M.any() and not V.any()


def test_gather_is_concatenation():
    rng = np.random.default_rng(13)
    sizes, unit_first = [4, 7, 2, 9, 5], [0, 2, 4]
    L = oracle.Layout(sizes, 3, unit_first)
    sh = [rng.integers(0, 1 << 16, size=L.shard_total, dtype=np.uint64).astype(np.uint16) for _ in range(3)]
    for u, U in enumerate(L.units):
        full = oracle.gather_unit(L, u, sh)
        assert full.size == U[3]
        want = np.concatenate([sh[r][U[6]:U[6] + U[4]] for r in range(3)])
        assert np.array_equal(full, want)


# ----------------------------------------------------------------- generator

def test_splitmix64_published_vectors():
    vals = []
    with open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                vals.append(int(line, 16))
    gamma = 0x9E3779B97F4A7C15
    assert [synth.hash64((k * gamma) % 2**64) for k in range(4)] == vals


def test_generator_statistics():
    w = W.workload(2)
    s = synth.grad_stream(w, 1, 0)
    h = s.host(0, 1 << 20)
    x = h.view(np.float16).astype(np.float64)
    base = synth.Stream(w.wid, W.KIND_GRAD, 1, 0, w.grad_sigma, w.dtype, False).host(0, 1 << 20)
    xb = base.view(np.float16).astype(np.float64)
    assert abs(xb.mean()) < 1e-4 and abs(xb.std() / 1e-2 - 1) < 1e-2
    assert np.abs(xb).max() <= 3.47e-2
    frac = np.mean(np.abs(x) > 0.0348)
    assert 0.008 < frac < 0.0102                   # 1 % outliers x100 (a few land below the cut)
    idx = np.array([0, 1, 5, 1 << 19, (1 << 20) - 1])
    assert np.array_equal(s.at(idx), h[idx])


def test_workload_shapes():
    """Parameter counts of the named model shapes (GPT-2 small 124,439,808; 1.3B GPT
    1,315,723,264; Llama-7B-shaped 6,738,415,616) and unit structure."""
    assert W.workload(0).phi == 1 << 20
    assert W.workload(2).phi == 124_439_808 and len(W.workload(2).sizes) == 148
    w3 = W.workload(3)
    assert w3.phi == 1_315_723_264 and len(w3.sizes) == 292 and len(w3.units()) == 26
    w4 = W.workload(4)
    assert w4.phi == 6_738_415_616 and len(w4.sizes) == 291 and len(w4.units()) == 34
    w1 = W.workload(1)
    assert len(w1.sizes) == 10000 and min(w1.sizes) >= 1 and max(w1.sizes) <= 65536
    assert 50e6 < w1.phi < 70e6


def test_scaler_trajectory():
    """Skip + halve on a flagged step (t unchanged); grow x2 after `interval` clean steps;
    never below the minimum scale."""
    cfg = W.Scaler(init_scale=8.0, growth_interval=3, min_scale=2.0)
    s = oracle.ScalerState(cfg)
    trace = []
    for flag in [0, 1, 0, 0, 0, 1, 1, 1, 0]:
        s.update(flag)
        trace.append((s.t, s.scale, s.good))
    assert trace == [(1, 8.0, 1), (1, 4.0, 0), (2, 4.0, 1), (3, 4.0, 2), (4, 8.0, 0),
                     (4, 4.0, 0), (4, 2.0, 0), (4, 2.0, 0), (5, 2.0, 1)]
    s = oracle.ScalerState(None)
    for flag in [0, 1, 0]:
        s.update(flag)
    assert (s.t, s.scale) == (2, 1.0)


# ----------------------------------------------------------------- gradient norm and clipping

def _oracle_run_1rank(gs16, p16, hyper, max_norm, is_fp16=0):
    """Run the sharded oracle with N_d = 1 over a sequence of 16-bit gradients."""
    n = p16.size
    L = oracle.Layout([n], 1)
    P = [oracle.widen16(p16, is_fp16).astype(np.float32)]
    M, V = [np.zeros(n, np.float32)], [np.zeros(n, np.float32)]
    full = p16.copy()
    norms = []
    for t, c in enumerate(gs16, start=1):
        k9 = oracle.consts(hyper, t, 1.0, 1)
        flag, n2 = oracle.sharded_step_ex(L, 1, 0, is_fp16, [c], [1], P, M, V, None, full, k9,
                                          max_norm)
        assert flag == 0
        norms.append(n2)
    return P[0], M[0], V[0], norms


def test_clipping_matches_torch():
    """Clip-by-global-norm then AdamW against torch.nn.utils.clip_grad_norm_ + torch AdamW
    (library cross-check of reading R8), with the clip active on every step."""
    hyper = W.Hyper()
    rng = np.random.default_rng(30)
    n = 5000
    p16 = _rand16(rng, n, 0, 0.02)
    gs = [_rand16(rng, n, 0, 0.01) for _ in range(4)]
    max_norm = 0.05                       # norm of ~N(0, 1e-2) over 5000 elements is ~0.7
    P, M, V, norms = _oracle_run_1rank(gs, p16, hyper, max_norm)
    tp = torch.nn.Parameter(torch.from_numpy(oracle.widen16(p16, 0).astype(np.float32)))
    opt = torch.optim.AdamW([tp], lr=hyper.lr, betas=(hyper.beta1, hyper.beta2), eps=hyper.eps,
                            weight_decay=hyper.weight_decay, foreach=False)
    for c, n2 in zip(gs, norms):
        tp.grad = torch.from_numpy(oracle.widen16(c, 0).astype(np.float32))
        tn = torch.nn.utils.clip_grad_norm_([tp], max_norm)
        assert abs(float(tn) - math.sqrt(n2)) <= 1e-6 * math.sqrt(n2)
        opt.step()
    st = opt.state[tp]
    for mine, ref in [(P, tp.detach().numpy()), (M, st["exp_avg"].numpy()), (V, st["exp_avg_sq"].numpy())]:
        assert np.all(np.abs(mine - ref) <= 1e-6 * np.abs(ref) + 1e-8)


def test_norm_and_coefficient_closed_forms():
    """Constant gradient c = 2^-7 over n = 4096 elements: norm^2 = n c^2 exactly, norm = 64 c;
    max_norm = 16 c gives coef = fp32(16c / (64c + 1e-6)) and m = fp32(0.1) * fp32(c * coef)."""
    hyper = W.Hyper()
    n, c = 4096, 2.0 ** -7
    g16 = oracle.round16(np.full(n, c, np.float32), 0)
    p16 = oracle.round16(np.zeros(n, np.float32), 0)
    P, M, V, norms = _oracle_run_1rank([g16], p16, hyper, 16 * c)
    assert fractions.Fraction(norms[0]) == n * fractions.Fraction(c) ** 2
    coef = np.float32(16 * c / (64 * c + 1e-6))
    assert oracle.clip_coef(norms[0], 16 * c) == coef
    assert np.all(M == np.float32(1 - hyper.beta1) * (np.float32(c) * coef))
    # a bound above the norm leaves the step bit-identical to the unclipped one
    P2, M2, V2, _ = _oracle_run_1rank([g16], p16, hyper, 1.0)
    P3, M3, V3, _ = _oracle_run_1rank([g16], p16, hyper, 0.0)
    assert np.array_equal(P2, P3) and np.array_equal(M2, M3) and np.array_equal(V2, V3)


def test_norm_is_exact_sum_of_squares():
    """Gradients that are small multiples of 2^-8: fp32(g*g) and their double sum are exact."""
    rng = np.random.default_rng(31)
    ints = rng.integers(-64, 65, size=777)
    g16 = oracle.round16((ints / 256.0).astype(np.float32), 0)
    _, _, _, norms = _oracle_run_1rank([g16], oracle.round16(np.zeros(777, np.float32), 0),
                                       W.Hyper(), 0.0)
    assert fractions.Fraction(norms[0]) == sum(fractions.Fraction(int(i), 256) ** 2 for i in ints)


# ----------------------------------------------------------------- FSDP-2 per-parameter sharding

def _random_pp_case(rng, max_tensors=8):
    nt = int(rng.integers(1, max_tensors + 1))
    dim0 = [int(x) for x in rng.integers(0, 9, size=nt)]
    cols = [int(x) for x in rng.integers(1, 5, size=nt)]
    sizes = [d * c for d, c in zip(dim0, cols)]
    units = []
    if nt > 1 and rng.random() < 0.6:
        cuts = sorted(set(int(x) for x in rng.integers(1, nt, size=int(rng.integers(1, 3)))))
        units = [0] + cuts
    return sizes, dim0, units


def test_per_param_chunks_brute_force():
    """Owner of element (tensor t, row i) = i // ceil(d0_t / N_d), by enumeration."""
    rng = np.random.default_rng(40)
    for _ in range(300):
        sizes, dim0, units = _random_pp_case(rng)
        n_d = int(rng.integers(1, 7))
        pp = oracle.PerParam(sizes, dim0, n_d, units)
        firsts = units or [0]
        unit_of = {t: max(i for i, f in enumerate(firsts) if f <= t) for t in range(len(sizes))}
        want, state = [], {r: 0 for r in range(n_d)}
        for r in range(n_d):
            for t in range(len(sizes)):
                u = unit_of[t]
                cols = sizes[t] // dim0[t] if dim0[t] else 0
                c_rows = -(-dim0[t] // n_d)
                owned = [i for i in range(dim0[t]) if i // c_rows == r] if c_rows else []
                unit_start = sum(sizes[firsts[u]:t])
                row0 = r * c_rows
                want.append((r, u, t, row0, len(owned), cols, c_rows, unit_start + row0 * cols, state[r]))
                assert not owned or owned[0] == row0
                state[r] += c_rows * cols
        assert [tuple(int(x) for x in row) for row in pp.chunks] == want
        assert all(state[r] == pp.per_rank for r in range(n_d))


def test_per_param_clipping_equals_the_flat_clipped_step():
    """R8 on per-parameter plans: the global norm and the clipping of the flat step (whose
    clipping is pinned to torch.nn.utils.clip_grad_norm_ above), over the same gradients.
    With every rank bound, norm^2 equals the flat step's up to the order of its double sum
    (1e-12 relative), and the owned rows of every rank's update, placed back, equal the flat
    step's update bit for bit whenever the two fp32 coefficients agree."""
    rng = np.random.default_rng(43)
    hyper = W.Hyper()
    clipped = 0
    for trial in range(120):
        sizes, dim0, units = _random_pp_case(rng)
        n = int(sum(sizes))
        if n == 0:
            continue
        n_d = int(rng.integers(1, 7))
        is_fp16 = int(rng.integers(0, 2))
        max_norm = float(rng.choice([1e-4, 1e-2, 1e3]))
        pp = oracle.PerParam(sizes, dim0, n_d, units)
        params16 = _rand16(rng, n, is_fp16, 0.02)
        contribs = [_rand16(rng, n, is_fp16) for _ in range(n_d)]
        k9 = oracle.consts(hyper, int(rng.integers(1, 5)), 1.0, n_d)
        p, m, v, sh = [], [], [], []
        for r in range(n_d):
            P = np.zeros(max(1, pp.per_rank), np.float32)
            S16 = np.zeros(max(1, pp.per_rank), np.uint16)
            for (rr, u, t, row0, rows, cols, c_rows, coff, soff) in pp.chunks:
                if rr == r and rows:
                    g0 = pp.unit_base[u] + coff
                    S16[soff:soff + rows * cols] = params16[g0:g0 + rows * cols]
                    P[soff:soff + rows * cols] = oracle.widen16(params16[g0:g0 + rows * cols], is_fp16)
            p.append(P)
            m.append(np.zeros_like(P))
            v.append(np.zeros_like(P))
            sh.append(S16)
        flag, n2pp = pp.step_ex(is_fp16, contribs, [1] * n_d, p, m, v, sh, k9, max_norm)
        assert flag == 0
        # the flat stage-1 step over the same tensors (padded to a multiple of N_d with zeros)
        L = oracle.Layout(sizes, n_d)
        pad = L.total_pad - n
        cf = [np.concatenate([c, np.zeros(pad, np.uint16)]) for c in contribs]
        pf16 = np.concatenate([params16, np.zeros(pad, np.uint16)])
        fp, fm, fv, fsh, full = [], [], [], [], pf16.copy()
        for r in range(n_d):
            U = L.units[0]
            seg = pf16[U[5] + r * U[4]:U[5] + (r + 1) * U[4]]
            fp.append(oracle.widen16(seg, is_fp16).astype(np.float32))
            fm.append(np.zeros(seg.size, np.float32))
            fv.append(np.zeros(seg.size, np.float32))
        f_flag, n2flat = oracle.sharded_step_ex(L, 1, 0, is_fp16, cf, [1] * n_d, fp, fm, fv, None, full,
                                                k9, max_norm)
        assert f_flag == 0
        assert abs(n2pp - n2flat) <= 1e-12 * n2flat, (trial, n2pp, n2flat)
        same_coef = oracle.clip_coef(n2pp, max_norm) == oracle.clip_coef(n2flat, max_norm)
        clipped += oracle.clip_coef(n2pp, max_norm) < 1.0
        Pf, Mf, Vf = _union(L, fp), _union(L, fm), _union(L, fv)
        for (r, u, t, row0, rows, cols, c_rows, coff, soff) in pp.chunks:
            g0 = pp.unit_base[u] + coff
            for mine, ref in ((p[r], Pf), (m[r], Mf), (v[r], Vf)):
                a, b = mine[soff:soff + rows * cols], ref[g0:g0 + rows * cols]
                if same_coef:
                    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), trial
                else:
                    assert np.all(np.abs(a - b) <= 1e-6 * np.abs(b) + 1e-8), trial
    assert clipped >= 30, clipped


def test_per_param_union_equals_ddp():
    """[ZF] 'Mathematical Formulation of ZeRO Partitioning Stages': per-parameter sharding also
    keeps data-parallel semantics -- the owned rows of every rank's update, placed back, equal
    the unsharded step bit for bit, and gathering the 16-bit shards rebuilds each unit."""
    rng = np.random.default_rng(41)
    hyper = W.Hyper()
    for trial in range(150):
        sizes, dim0, units = _random_pp_case(rng)
        n_d = int(rng.integers(1, 7))
        is_fp16 = int(rng.integers(0, 2))
        pp = oracle.PerParam(sizes, dim0, n_d, units)
        n = int(sum(sizes))
        params16 = _rand16(rng, n, is_fp16, 0.02)
        contribs = [_rand16(rng, n, is_fp16) for _ in range(n_d)]
        k9 = oracle.consts(hyper, int(rng.integers(1, 5)), 1.0, n_d)
        p, m, v, sh = [], [], [], []
        for r in range(n_d):
            P = np.zeros(max(1, pp.per_rank), np.float32)
            S16 = np.zeros(max(1, pp.per_rank), np.uint16)
            for (rr, u, t, row0, rows, cols, c_rows, coff, soff) in pp.chunks:
                if rr == r and rows:
                    g0 = pp.unit_base[u] + coff
                    S16[soff:soff + rows * cols] = params16[g0:g0 + rows * cols]
                    P[soff:soff + rows * cols] = oracle.widen16(params16[g0:g0 + rows * cols], is_fp16)
            p.append(P)
            m.append(np.zeros_like(P))
            v.append(np.zeros_like(P))
            sh.append(S16)
        assert pp.step(is_fp16, contribs, [1] * n_d, p, m, v, sh, k9) == 0
        Pd = oracle.widen16(params16, is_fp16).astype(np.float32)
        Md, Vd = np.zeros(n, np.float32), np.zeros(n, np.float32)
        out = np.zeros(n, np.uint16)
        assert oracle.ddp_step(contribs, is_fp16, Pd, Md, Vd, out, k9) == 0
        for (r, u, t, row0, rows, cols, c_rows, coff, soff) in pp.chunks:
            g0 = pp.unit_base[u] + coff
            for mine, ref in ((p[r], Pd), (m[r], Md), (v[r], Vd)):
                assert np.array_equal(mine[soff:soff + rows * cols].view(np.uint32),
                                      ref[g0:g0 + rows * cols].view(np.uint32)), trial
        for u in range(len(pp.unit_numel)):
            lo = pp.unit_base[u]
            assert np.array_equal(pp.gather(u, sh), out[lo:lo + pp.unit_numel[u]])
