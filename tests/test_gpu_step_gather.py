"""GPU parity of the step launch that also streams the next unit's all-gather
(zero_step_gather_next, and zero_step_units_overlapped with one stream).

Per step: unit 0 is gathered on its own, then every launch runs unit u's fused reduce +
AdamW + cast and, after its tiles, gathers unit u+1 into the other of two buffers.  Checked
against the oracle on the same seeded inputs: every gathered unit bit for bit (the gather
reads the shards the previous step wrote), the fp32 state within 1e-6 |x| + 1e-8, the 16-bit
shards within 1 ulp, skips, t and the loss scale exactly.  Also: the register-load fallback
(gather as a launch of its own), per-parameter plans (the wide parameter block), a tiny step
carrying a large gather, clipping, norm-report steps (which fall back), the one-stream
schedule (also captured in a CUDA graph and replayed), the 1.3B and Llama workloads sampled at
full size, flat and per-parameter, and a wait that runs out inside the gather part.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gpu_harness as H
import synth
import zero_sharded_mixed_03_gb300 as Z
from synth import workloads as W

pytestmark = pytest.mark.gpu

BULK = {Z.ZERO_OPT_STAGING: Z.ZERO_STAGING_BULK}
LDG = {Z.ZERO_OPT_STAGING: Z.ZERO_STAGING_REGISTER_LOADS}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    Z.lib()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _mk(wid, sizes, n_d, steps=3, units=(), dtype=W.BF16, scaler=None, inject=None, bound=None):
    return W.Workload(wid=wid, name=f"sg{wid}", sizes=tuple(sizes), n_d=n_d, stage=3,
                      bucket_elems=0, unit_first=tuple(units), dtype=dtype, steps=steps,
                      hyper=W.Hyper(), scaler=scaler, inject=inject, bound_ranks=bound)


def _ragged(seed, n, hi):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1, hi, size=n)]


def _pp(wid, n_t, n_d, seed, units, max_rows=300, max_cols=64, bound=None):
    rng = np.random.default_rng(seed)
    dim0 = [int(x) for x in rng.integers(1, max_rows, size=n_t)]
    sizes = [d * int(c) for d, c in zip(dim0, rng.integers(1, max_cols, size=n_t))]
    return W.Workload(wid=wid, name=f"sgpp{wid}", sizes=tuple(sizes), n_d=n_d, stage=3,
                      bucket_elems=0, unit_first=tuple(units), dtype=W.BF16, steps=3,
                      hyper=W.Hyper(), scaler=None, bound_ranks=bound, dim0=tuple(dim0),
                      per_param=True)


CASES = {
    "nd16_units": _mk(501, _ragged(4, 24, 60000), 16, units=(0, 5, 11, 17, 23)),
    # ragged shards (heads and tails in the gather copies), peers, fp16, a skipped first step
    "nd3_fp16_peers_skip_first": _mk(502, _ragged(5, 12, 30000), 3, units=(0, 4, 9),
                                     dtype=W.FP16, scaler=W.Scaler(init_scale=1024.0),
                                     inject=(1, 2, 1234), bound=(0, 2)),
    # a tiny unit's step carrying a large unit's gather (more gather chunks than tiles)
    "nd8_tiny_step_big_gather": _mk(503, [40, 3, 2_000_003, 1_500_000, 7], 8, units=(0, 2, 4)),
    "nd7_odd_shards": _mk(504, [1_000_001, 333_333, 77_777, 5], 7, units=(0, 1, 3)),
    # more than 32 gather copies: the wide parameter block
    "pp_nd16_wide": _pp(505, 30, 16, 3, units=(0, 10, 20), max_rows=400),
    "pp_nd8_peers": _pp(506, 16, 8, 2, units=(0, 5, 9), bound=(0, 3, 7)),
}


def _fill_units(run, w, k, contribs):
    for u, (which, lo, hi) in enumerate(run.ranges()):
        for r in range(w.n_d):
            H.fill_device(contribs[u][r], synth.grad_stream(w, k, r), run.units, lo, hi)


def _run_fused(w, options=None, expect_fused=True, check_norm=False):
    run = H.Run(w, options=options, alloc_contribs=False)
    o = H.OracleFull(w, run.bound)
    nu = len(run.units)
    maxu = int(run.info.max_unit_pad)
    bufs = [torch.empty(max(8, maxu), dtype=torch.int16, device="cuda") for _ in range(2)]
    contribs = [[torch.empty(max(8, U[3]), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
                for U in run.units]
    in_step = []
    try:
        for k in range(1, w.steps + 1):
            expect_g = [o.gathered(u) for u in range(nu)]
            _fill_units(run, w, k, contribs)
            if w.hyper.max_grad_norm > 0:              # clipping: the norm over every unit first
                for u in range(nu):
                    run.g.grad_norm([c.data_ptr() for c in contribs[u]], u)
            run.g.gather(0, bufs[0])
            for u in range(nu):
                torch.cuda.synchronize()
                n = run.units[u][3]
                got = bufs[u % 2][:n].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, expect_g[u]), f"gathered unit {u} at step {k}"
                run.g.release(u)
                ptrs = [c.data_ptr() for c in contribs[u]]
                if u + 1 < nu:
                    run.g.step_gather_next(ptrs, u, run.hyper, u + 1, bufs[(u + 1) % 2])
                    in_step.append(Z.zero_get_option(run.g.plan, Z.ZERO_OPT_LAST_GATHER_IN_STEP))
                else:
                    run.g.step(ptrs, u, run.hyper)
            res = run.g.finish()
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale, f"step {k}"
            H.compare_full(run, o, f"{w.name} fused step {k}")
            if check_norm:
                want = float(np.sqrt(o.norm2))
                assert abs(res.grad_norm - want) <= 1e-12 * want, (res.grad_norm, want)
        if expect_fused is not None:
            assert all(x == (1 if expect_fused else 0) for x in in_step), in_step
        return in_step
    finally:
        run.close()


@pytest.mark.parametrize("name", list(CASES))
def test_step_with_next_gather_full_parity(name):
    _run_fused(CASES[name], options=BULK)


@pytest.mark.parametrize("name", ["nd16_units", "nd7_odd_shards"])
def test_step_with_next_gather_automatic_choice(name):
    _run_fused(CASES[name])


def test_step_with_next_gather_tiny_case_sweep():
    """Bounds of the gather part: 60 random stage-3 plans, flat (phi <= 120) and per-parameter
    (dim-0 rows <= 20), N_d 1..16, bf16 and fp16, zero-size tensors, random subsets of the
    ranks bound; every unit gathered inside the previous unit's step launch where the kernel
    takes it; two steps each against the oracle."""
    rng = np.random.default_rng(62)
    fused = 0
    for trial in range(60):
        nt = int(rng.integers(1, 8))
        n_d = int(rng.integers(1, 17))
        units = tuple([0] + sorted(set(int(x) for x in rng.integers(1, nt, size=3)))) if nt > 1 else (0,)
        bound = None
        if n_d > 1 and rng.integers(0, 2):
            bound = tuple(sorted(set(int(x) for x in rng.integers(0, n_d, size=int(rng.integers(1, n_d))))))
        dtype = int(rng.integers(0, 2))
        if trial % 2:
            dim0 = [int(x) for x in rng.integers(0, 21, size=nt)]
            sizes = [d * int(c) for d, c in zip(dim0, rng.integers(1, 9, size=nt))]
            w = W.Workload(wid=700 + trial, name=f"sgtiny{trial}", sizes=tuple(sizes), n_d=n_d,
                           stage=3, bucket_elems=0, unit_first=units, dtype=dtype, steps=2,
                           hyper=W.Hyper(), scaler=None, bound_ranks=bound, dim0=tuple(dim0),
                           per_param=True)
        else:
            sizes = [int(x) for x in rng.integers(0, 21, size=nt)]
            if sum(sizes) == 0:
                sizes[0] = 1
            w = dataclasses.replace(_mk(700 + trial, sizes, n_d, steps=2, units=units, bound=bound),
                                    dtype=dtype)
        fused += any(_run_fused(w, options=BULK, expect_fused=None))
    assert fused >= 20, fused                  # most plans take the gather into the launch


@pytest.mark.parametrize("name", ["nd16_units", "nd3_fp16_peers_skip_first", "pp_nd8_peers"])
def test_step_with_next_gather_register_loads_fallback(name):
    """With the register-load step kernel the gather runs as a launch of its own: same results."""
    _run_fused(CASES[name], options=LDG, expect_fused=False)


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("name", ["nd16_units", "nd3_fp16_peers_skip_first", "pp_nd16_wide"])
def test_one_stream_overlapped_schedule(name, order):
    """zero_step_units_overlapped without a second stream: the gathers run inside the steps;
    states, shards and the last two gathered units (left in the buffers) match the oracle.
    Units first to last, and last to first (ZERO_OPT_UNIT_ORDER = 1: a backward pass's order)."""
    w = CASES[name]
    run = H.Run(w, options={**BULK, Z.ZERO_OPT_UNIT_ORDER: order}, alloc_contribs=False)
    o = H.OracleFull(w, run.bound)
    nu = len(run.units)
    maxu = int(run.info.max_unit_pad)
    bufs = [torch.empty(max(8, maxu), dtype=torch.int16, device="cuda") for _ in range(2)]
    contribs = [[torch.empty(max(8, U[3]), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
                for U in run.units]
    try:
        for k in range(1, w.steps + 1):
            expect_g = [o.gathered(u) for u in range(nu)]
            _fill_units(run, w, k, contribs)
            ptrs = [c.data_ptr() for unit in contribs for c in unit]
            res = Z.zero_step_units_overlapped(run.g.plan, ptrs, [b.data_ptr() for b in bufs],
                                               run.hyper, torch.cuda.current_stream().cuda_stream,
                                               None)
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale
            torch.cuda.synchronize()
            seq = list(range(nu))[::-1] if order else list(range(nu))
            for i in range(max(0, nu - 2), nu):            # the last two positions of the order
                u = seq[i]
                got = bufs[i % 2][:run.units[u][3]].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, expect_g[u]), f"gathered unit {u} at step {k}"
            H.compare_full(run, o, f"one-stream {name} order {order} step {k}")
    finally:
        run.close()


@pytest.mark.parametrize("cfg,per_param,bound", [(3, False, None), (4, False, (0, 7)),
                                                  (3, True, None), (4, True, (0, 7))])
def test_step_with_next_gather_config_sampled(cfg, per_param, bound):
    """The ZeRO-3 1.3B and Llama rank-view workloads at full size (flat and per-parameter
    plans) in the one-stream schedule the bench times: sampled state elements and every
    gathered unit at sampled positions against the oracle."""
    w = W.workload(cfg)
    if per_param:
        w = W.per_param_variant(w)
    w = dataclasses.replace(w, steps=2)
    run = H.Run(w, bound=bound, options=BULK)
    try:
        idx = H.sample_indices(run, 20000)
        o = H.OracleSampled(w, idx)
        # elements of ranks without local state: their gathered values stay the initial ones
        allr = H.sample_indices(run, 4000, seed=1, bound_only=False)
        rank, _ = run.locate(allr)
        peer_idx = allr[rank < 0]
        peer16 = H.values_at(synth.param_stream(w), o.units, peer_idx)
        nu = len(run.units)
        maxu = int(run.info.max_unit_pad)
        bufs = [torch.empty(maxu, dtype=torch.int16, device="cuda") for _ in range(2)]
        calls = run.ranges()
        for k in range(1, w.steps + 1):
            exp_idx = np.concatenate([idx, peer_idx])
            exp16 = np.concatenate([o.out16, peer16])    # the shards the previous step left
            run.g.gather(0, bufs[0])
            for u, (which, lo, hi) in enumerate(calls):
                torch.cuda.synchronize()
                sel = (exp_idx >= lo) & (exp_idx < hi)
                if sel.any():
                    got = bufs[u % 2][torch.from_numpy(exp_idx[sel] - lo).cuda()].cpu().numpy().view(np.uint16)
                    assert np.array_equal(got, exp16[sel]), f"gathered unit {u} at step {k}"
                run.g.release(u)
                for r in range(w.n_d):
                    H.fill_device(run.contribs[r], synth.grad_stream(w, k, r), run.units, lo, hi)
                ptrs = [c.data_ptr() for c in run.contribs]
                if u + 1 < nu:
                    run.g.step_gather_next(ptrs, u, run.hyper, u + 1, bufs[(u + 1) % 2])
                    assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_LAST_GATHER_IN_STEP) == 1
                else:
                    run.g.step(ptrs, u, run.hyper)
            res = run.g.finish()
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t, f"step {k}"
            st, g16 = run.read_sampled(idx)
            for key, want in (("master", o.p), ("m", o.m), ("v", o.v)):
                H.assert_state_close(st[key], want, f"{w.name} fused step {k} {key}")
            H.assert_16_close(g16, o.out16, f"{w.name} fused step {k} 16-bit")
    finally:
        run.close()


def test_step_with_next_gather_argument_errors():
    w = CASES["nd7_odd_shards"]
    run = H.Run(w, options=BULK)
    try:
        buf = torch.empty(int(run.info.max_unit_pad), dtype=torch.int16, device="cuda")
        ptrs = [c.data_ptr() for c in run.contribs]
        for bad_next in (0, -1, len(run.units)):                  # the stepped unit, out of range
            with pytest.raises(Z.ZeroError) as e:
                run.g.step_gather_next(ptrs, 0, run.hyper, bad_next, buf)
            assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:                      # the whole step: it would
            run.g.step_gather_next(ptrs, -1, run.hyper, 1, buf)    # update unit 1 as it gathers
        assert e.value.status == Z.ZERO_EINVAL
        run.g.gather(1, buf)
        with pytest.raises(Z.ZeroError) as e:                      # still gathered
            run.g.step_gather_next(ptrs, 0, run.hyper, 1, buf)
        assert e.value.status == Z.ZERO_ESTATE
        run.g.release(1)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_step_gather_next(run.g.plan, ptrs, 0, run.hyper, 1, 0)
        assert e.value.status == Z.ZERO_EINVAL                     # NULL destination
        torch.cuda.synchronize()
    finally:
        run.close()


def test_wait_limit_runs_out_in_the_gather_part():
    """With a wait limit of 0 the first barrier wait that is not already satisfied gives up,
    in the step tiles or in the gather chunks: the kernel records it, drains its copies and
    returns, the step is discarded (ZERO_ETIMEOUT, state unchanged), and the next step with
    the normal limit follows the oracle."""
    w = _mk(507, [3_000_000 + 5, 2_500_000, 17], 4, steps=2, units=(0, 1))
    run = H.Run(w, options=BULK, alloc_contribs=False)
    o = H.OracleFull(w, run.bound)
    bufs = [torch.empty(int(run.info.max_unit_pad), dtype=torch.int16, device="cuda") for _ in range(2)]
    contribs = [[torch.empty(max(8, U[3]), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
                for U in run.units]

    def step(k):
        _fill_units(run, w, k, contribs)
        run.g.gather(0, bufs[0])
        run.g.release(0)
        run.g.step_gather_next([c.data_ptr() for c in contribs[0]], 0, run.hyper, 1, bufs[1])
        run.g.release(1)
        run.g.step([c.data_ptr() for c in contribs[1]], 1, run.hyper)
        return run.g.finish()

    try:
        res = step(1)
        o.step(1)
        assert res.t == 1
        before = {r: run.read_logical(r) for r in run.bound}
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 0)
        with pytest.raises(Z.ZeroError) as e:
            step(2)
        assert e.value.status == Z.ZERO_ETIMEOUT
        st = e.value.result
        assert (st.t, st.finished) == (1, 1)
        for r in run.bound:
            now = run.read_logical(r)
            for key in now:
                assert np.array_equal(now[key].view(np.uint32), before[r][key].view(np.uint32)), key
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 1_000_000_000)
        res = step(2)
        o.step(2)
        assert (res.t, res.finished, res.skipped) == (2, 2, 0)
        H.compare_full(run, o, "after the timeout")
    finally:
        run.close()


def test_step_with_next_gather_edge_units():
    """An empty unit as the next one (nothing to gather), and a per-parameter unit whose gather
    has more copies (20 tensors x 16 ranks) than the wide parameter block holds: that launch
    runs its gather separately, the others inside; results match the oracle either way."""
    empty_next = _mk(511, [0, 40, 0, 0, 33, 1, 0], 16, units=(0, 2, 4))
    _run_fused(empty_next, options=BULK, expect_fused=None)
    many = _pp(512, 24, 16, 9, units=(0, 2, 22), max_rows=600)
    _run_fused(many, options=BULK, expect_fused=None)


def test_step_with_next_gather_and_clipping():
    """Clipping (norm pre-pass over every unit, then the clip-mode step): the step launches
    still carry the next unit's gather; states and the norm match the oracle."""
    w = dataclasses.replace(CASES["nd16_units"], wid=508, hyper=W.Hyper(max_grad_norm=0.02))
    _run_fused(w, options=BULK, check_norm=True)


def test_step_with_next_gather_norm_report_falls_back():
    """Norm-report steps run the register-load kernel, so the gather is a launch of its own;
    the update is unchanged and the reported norm matches the oracle."""
    w = dataclasses.replace(CASES["nd16_units"], wid=509, hyper=W.Hyper(report_norm=True))
    _run_fused(w, options=BULK, expect_fused=False, check_norm=True)


def test_one_stream_schedule_captured_in_a_cuda_graph():
    """A whole one-stream step (unit 0's gather, the step launches that gather the next unit,
    the re-cast and the commit) captured once and replayed with new gradients written in place:
    every replay follows the oracle, through a skipped step."""
    w = dataclasses.replace(CASES["nd3_fp16_peers_skip_first"], wid=510, steps=4, inject=(3, 1, 4321))
    run = H.Run(w, options=BULK, alloc_contribs=False)
    o = H.OracleFull(w, run.bound)
    nu = len(run.units)
    bufs = [torch.empty(int(run.info.max_unit_pad), dtype=torch.int16, device="cuda") for _ in range(2)]
    contribs = [[torch.empty(max(8, U[3]), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
                for U in run.units]
    ptrs = [c.data_ptr() for unit in contribs for c in unit]
    gptrs = [b.data_ptr() for b in bufs]

    def enqueue(stream):
        Z.zero_step_units_overlapped(run.g.plan, ptrs, gptrs, run.hyper, stream.cuda_stream, None,
                                     wait=False)

    try:
        _fill_units(run, w, 1, contribs)
        enqueue(torch.cuda.current_stream())      # step 1 uncaptured: bias table, kernel set-up
        o.step(1)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                enqueue(side)                     # captured, not run
        skips = 0
        for k in range(2, w.steps + 1):
            expect_last = o.gathered(nu - 1)
            _fill_units(run, w, k, contribs)
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            skips += o.step(k)
            st = run.g.step_state()
            assert (st.t, st.scale, st.skipped_total) == (o.sc.t, o.sc.scale, skips), k
            got = bufs[(nu - 1) % 2][:run.units[nu - 1][3]].cpu().numpy().view(np.uint16)
            assert np.array_equal(got, expect_last), f"gathered unit {nu - 1} at replay {k}"
            H.compare_full(run, o, f"one-stream graph replay step {k}")
        assert skips == 1
    finally:
        run.close()
