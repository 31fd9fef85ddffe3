"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs.

Tolerances (fp32 master/m/v): |gpu - oracle| <= 1e-6 |oracle| + 1e-8; 16-bit params: <= 1 ulp;
tables, skip decisions, step counts and loss scales: exact.
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


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    Z.lib()   # the product library must load; no fallback exists
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _mk(wid, sizes, n_d, stage, steps=3, bucket=0, units=(), dtype=W.BF16, scaler=None,
        outliers=False, inject=None, bound=None):
    return W.Workload(wid=wid, name=f"case{wid}", sizes=tuple(sizes), n_d=n_d, stage=stage,
                      bucket_elems=bucket, unit_first=tuple(units), dtype=dtype, steps=steps,
                      hyper=W.Hyper(), scaler=scaler, outliers=outliers, inject=inject,
                      bound_ranks=bound)


def _ragged(seed, n, hi):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1, hi, size=n)]


SMALL_CASES = {
    "z1_nd4_tiles_ragged_tail": _mk(101, [3 * 65536 + 13], 4, 1),
    "z2_nd7_ragged_tensors": _mk(102, _ragged(1, 60, 5000), 7, 2, steps=4),
    "z2_nd8_fp16_buckets_inf": _mk(103, _ragged(2, 40, 9000), 8, 2, steps=4, bucket=10_000,
                                   dtype=W.FP16, scaler=W.Scaler(), outliers=True,
                                   inject=(2, 3, 77_777)),
    "z2_nd5_odd_bucket_scalar_path": _mk(104, _ragged(3, 30, 7000), 5, 2, bucket=12_345),
    "z3_nd16_units": _mk(105, _ragged(4, 24, 6000), 16, 3, units=(0, 5, 11, 17, 23)),
    "z3_nd3_fp16_peers_skip_first": _mk(106, _ragged(5, 12, 3000), 3, 3, units=(0, 4, 9),
                                        dtype=W.FP16, scaler=W.Scaler(init_scale=1024.0),
                                        inject=(1, 2, 1234), bound=(0, 2)),
    "z1_nd1": _mk(107, [1000, 1], 1, 1),
    "z2_nd40_many_segments": _mk(108, _ragged(6, 50, 9000), 40, 2, bucket=4096),
    "z2_nd20_rank_batches": _mk(109, _ragged(7, 20, 20000), 20, 2),
    "z2_tiny_shard_below_vector": _mk(110, [5], 3, 2),
    "z3_nd16_fp16": _mk(111, _ragged(8, 16, 12000), 16, 3, units=(0, 3, 8), dtype=W.FP16),
    "z2_nd8_subset_bound": _mk(112, _ragged(9, 25, 8000), 8, 2, bucket=8000, bound=(1, 6)),
    "z3_nd16_empty_unit_tensors": _mk(113, [0, 40, 0, 0, 33, 1, 0], 16, 3, units=(0, 2, 4)),
}


def _compare_full(run: H.Run, o: H.OracleFull, label: str):
    return H.compare_full(run, o, label)


def _run_full(w: W.Workload, options=None):
    run = H.Run(w, options=options)
    o = H.OracleFull(w, run.bound)
    mism = 0
    try:
        for k in range(1, w.steps + 1):
            expect_g = [o.gathered(u) for u in range(len(o.units))] if w.stage == 3 else None

            def check(u, lo, hi, buf):
                got = buf[:hi - lo].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, expect_g[u]), f"gather of unit {u} at step {k}"

            res = run.step(k, check if w.stage == 3 else None)
            flag = o.step(k)
            assert res.skipped == flag, f"step {k}"
            assert res.t == o.sc.t and res.scale == o.sc.scale, f"step {k}"
            mism += _compare_full(run, o, f"{w.name} step {k}")
    finally:
        run.close()
    return mism


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_small_case_full_parity(name):
    _run_full(SMALL_CASES[name])


# N_d at its limit (ZERO_MAX_RANKS = 128 contribution pointers in the kernel parameters):
# ZeRO-2 over ragged tensors with buckets, and ZeRO-3 with an fp16 skip; both kernels.
MAX_RANK_CASES = {
    "z2_nd128_buckets": _mk(190, _ragged(30, 12, 40000), 128, 2, steps=2, bucket=50_000),
    "z3_nd128_fp16_skip": _mk(191, _ragged(31, 9, 30000), 128, 3, steps=3, units=(0, 4),
                              dtype=W.FP16, scaler=W.Scaler(init_scale=2048.0),
                              inject=(2, 77, 5), bound=(0, 64, 127)),
}


@pytest.mark.parametrize("staging", [0, 1])
@pytest.mark.parametrize("name", list(MAX_RANK_CASES))
def test_max_ranks_full_parity(name, staging):
    _run_full(MAX_RANK_CASES[name], options={Z.ZERO_OPT_STAGING: staging})


def test_config0_full_parity():
    w = W.workload(0)
    mism = _run_full(w)
    print(f"{w.name}: {mism} bit mismatches (within tolerance)")


def _run_sampled(w: W.Workload, bound=None, n_random=20000, options=None):
    run = H.Run(w, bound=bound, options=options)
    try:
        idx = H.sample_indices(run, n_random)
        o = H.OracleSampled(w, idx)
        peer_idx, peer16 = None, None
        if w.stage == 3:
            # elements of ranks without local state: the gather must return their initial values
            allr = H.sample_indices(run, 4000, seed=1, bound_only=False)
            rank, _ = run.locate(allr)
            peer_idx = allr[rank < 0]
            peer16 = H.values_at(synth.param_stream(w), o.units, peer_idx)
        mism = 0
        for k in range(1, w.steps + 1):
            if w.stage == 3:
                exp_idx = np.concatenate([idx, peer_idx])
                exp16 = np.concatenate([o.out16, peer16])

            def check(u, lo, hi, buf):
                sel = (exp_idx >= lo) & (exp_idx < hi)
                if sel.any():
                    got = buf[torch.from_numpy(exp_idx[sel] - lo).cuda()].cpu().numpy().view(np.uint16)
                    assert np.array_equal(got, exp16[sel]), f"gather unit {u} step {k}"

            res = run.step(k, check if w.stage == 3 else None)
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale, f"step {k}"
            st, g16 = run.read_sampled(idx)
            for key, want in (("master", o.p), ("m", o.m), ("v", o.v)):
                mism += H.assert_state_close(st[key], want, f"{w.name} step {k} {key}")
            mism += H.assert_16_close(g16, o.out16, f"{w.name} step {k} 16-bit")
        return idx.size, mism
    finally:
        run.close()


@pytest.mark.parametrize("i", [1, 2, 3])
def test_config_sampled_parity(i):
    n, mism = _run_sampled(W.workload(i))
    print(f"{W.workload(i).name}: {n} sampled elements, {mism} bit mismatches (within tolerance)")


@pytest.mark.parametrize("i,steps", [(1, 64), (2, 40)])
def test_config_sampled_long_run(i, steps):
    """Many steps at full size (the ragged ZeRO-2 workload; the fp16 GPT-2 workload with its
    loss scale and the skipped step 3): sampled state, parameters, t, skips and the scale
    after every step, so that nothing drifts as the bias correction and the moments evolve."""
    w = dataclasses.replace(W.workload(i), steps=steps)
    n, mism = _run_sampled(w)
    print(f"{w.name}, {steps} steps: {n} sampled elements, {mism} bit mismatches (within tolerance)")


def test_config4_rank0_and_last_rank_sampled():
    w = W.workload(4)
    n, mism = _run_sampled(w, bound=(0, w.n_d - 1))
    print(f"{w.name}, ranks 0 and {w.n_d - 1}: {n} sampled elements, {mism} bit mismatches")


# ---------------------------------------------------------------------- guards and errors

def test_guard_bands_and_layout_gaps_untouched():
    """Buffers embedded in larger ones filled with a canary: nothing outside the plan's
    elements (and nothing in the layout's phase gaps) may change."""
    sizes = _ragged(11, 30, 5000)
    n_d, G = 7, 256
    plan = Z.zero_plan_create(sizes, n_d, 3, 0, [0, 9, 19], Z.ZERO_BF16)
    try:
        rows = Z.zero_plan_tables(plan, Z.ZERO_TABLE_STATE_LAYOUT)
        units = Z.zero_plan_tables(plan, Z.ZERO_TABLE_UNITS)
        canary_f = np.float32(np.frombuffer(np.uint32(0x7FBADBAD).tobytes(), np.float32)[0])
        big, views, sh = {}, {}, {}
        for r in range(n_d):
            n = Z.zero_rank_state_elems(plan, r)
            b = torch.full((6, n + 2 * G), 0, dtype=torch.float32, device="cuda")
            b.view(torch.int32).fill_(0x7FBADBAD)
            s16 = torch.full((n + 2 * G,), 0x5A5A, dtype=torch.int16, device="cuda")
            big[r], sh[r] = b, s16
            for (rr, u, off, cnt) in rows:
                if rr == r:
                    b[:, G + off:G + off + cnt] = 0.0
                    b[0, G + off:G + off + cnt] = 0.01
                    s16[G + off:G + off + cnt] = 0
            views[r] = [b[j, G:G + n] for j in range(6)]
        ws = torch.zeros(Z.zero_plan_info(plan).workspace_bytes // 4, dtype=torch.int32, device="cuda")
        for r in range(n_d):
            v = views[r]
            Z.zero_bind(plan, r, [v[0].data_ptr(), v[1].data_ptr()], [v[2].data_ptr(), v[3].data_ptr()],
                        [v[4].data_ptr(), v[5].data_ptr()], sh[r][G:].data_ptr(), None, ws.data_ptr())
        maxc = Z.zero_plan_info(plan).max_contrib_elems
        contribs = [torch.full((maxc,), 0x3C00, dtype=torch.int16, device="cuda") for _ in range(n_d)]
        gbuf = torch.full((maxc + 2 * G,), 0x1234, dtype=torch.int16, device="cuda")
        for u, U in enumerate(units):
            Z.zero_gather_layer(plan, u, gbuf[G:].data_ptr())
            Z.zero_release_layer(plan, u)
            assert (gbuf[:G] == 0x1234).all() and (gbuf[G + U[3]:] == 0x1234).all()
            Z.zero_step(plan, [c.data_ptr() for c in contribs], u, Z.hyper())
        res = Z.zero_step_finish(plan)
        assert res.skipped == 0 and res.t == 1
        torch.cuda.synchronize()
        for r in range(n_d):
            b = big[r].view(torch.int32).cpu().numpy()
            s16 = sh[r].cpu().numpy()
            mask = np.ones(b.shape[1], dtype=bool)
            for (rr, u, off, cnt) in rows:
                if rr == r:
                    mask[G + off:G + off + cnt] = False
            assert (b[:, mask] == 0x7FBADBAD).all(), f"rank {r} state guard/gap overwritten"
            assert (s16[mask] == 0x5A5A).all(), f"rank {r} shard16 guard/gap overwritten"
            assert not (b[0, ~mask] == 0x7FBADBAD).any()
    finally:
        Z.zero_plan_destroy(plan)


def test_misaligned_contributions_take_the_scalar_path():
    """Contribution views starting one element past a 16-byte boundary: same results."""
    w = _mk(120, _ragged(12, 20, 4000), 4, 2, steps=2)
    ref = H.Run(w)
    alt = H.Run(w)
    try:
        for k in (1, 2):
            ref.step(k)
            for which, lo, hi in alt.ranges():
                for r in range(w.n_d):
                    H.fill_device(alt.contribs[r], synth.grad_stream(w, k, r),
                                  alt.units, lo, hi)
                shifted = []
                for c in alt.contribs:
                    s = torch.empty(c.numel() + 1, dtype=torch.int16, device="cuda")
                    s[1:] = c
                    shifted.append(s)
                alt.g.step([s[1:].data_ptr() for s in shifted], which, alt.hyper)
                torch.cuda.synchronize()
            alt.g.finish()
        for r in ref.bound:
            a, b = ref.read_logical(r), alt.read_logical(r)
            for key in a:
                assert np.array_equal(a[key].view(np.uint32), b[key].view(np.uint32))
        assert torch.equal(ref.g.full16, alt.g.full16)
    finally:
        ref.close()
        alt.close()


def test_step_lifecycle_errors():
    w = _mk(121, [1000, 2000], 2, 2, bucket=1000)
    run = H.Run(w)
    try:
        ptrs = [c.data_ptr() for c in run.contribs]
        run.g.step(ptrs, 0, run.hyper)
        with pytest.raises(Z.ZeroError) as e:
            run.g.step(ptrs, 0, run.hyper)            # bucket twice in one step
        assert e.value.status == Z.ZERO_ESTATE
        with pytest.raises(Z.ZeroError) as e:
            run.g.finish()                              # buckets 1, 2 missing
        assert e.value.status == Z.ZERO_ESTATE
        with pytest.raises(Z.ZeroError) as e:
            run.g.step(ptrs, 1, Z.hyper(lr=2e-3))       # hyperparameters changed mid-step
        assert e.value.status == Z.ZERO_EINVAL
        run.g.step(ptrs, 1, run.hyper)
        run.g.step(ptrs, 2, run.hyper)
        assert run.g.finish().t == 1
        with pytest.raises(Z.ZeroError) as e:
            run.g.step(ptrs, -2, run.hyper)
        assert e.value.status == Z.ZERO_EINVAL
    finally:
        run.close()


def test_empty_model_step():
    plan = Z.zero_plan_create([], 3, 2, 0, None, Z.ZERO_BF16)
    try:
        ws = torch.zeros(Z.zero_plan_info(plan).workspace_bytes // 4, dtype=torch.int32, device="cuda")
        dummy = torch.zeros(8, dtype=torch.float32, device="cuda")
        d2 = torch.zeros(8, dtype=torch.float32, device="cuda")
        f16 = torch.zeros(8, dtype=torch.int16, device="cuda")
        Z.zero_bind(plan, 0, [dummy.data_ptr(), d2.data_ptr()], [dummy.data_ptr() + 4, d2.data_ptr() + 4],
                    [dummy.data_ptr() + 8, d2.data_ptr() + 8], None, f16.data_ptr(), ws.data_ptr())
        Z.zero_step(plan, [f16.data_ptr()] * 3, -1, Z.hyper())
        res = Z.zero_step_finish(plan)
        assert res.skipped == 0 and res.t == 1
    finally:
        Z.zero_plan_destroy(plan)


# ---------------------------------------------------------------------- device-resident step state

def test_steps_enqueued_without_host_waits():
    """Five steps (one with a planted inf) enqueued back to back, the commit left on the device:
    one read-back at the end must match the oracle's state, t, loss scale and skip count."""
    w = _mk(130, _ragged(13, 30, 6000), 6, 2, steps=5, bucket=9_000, dtype=W.FP16,
            scaler=W.Scaler(init_scale=4096.0, growth_interval=2), inject=(3, 4, 5_000))
    run = H.Run(w)
    o = H.OracleFull(w, run.bound)
    try:
        for k in range(1, w.steps + 1):
            for which, lo, hi in run.ranges():
                for r in range(w.n_d):
                    H.fill_device(run.contribs[r], synth.grad_stream(w, k, r), run.units, lo, hi)
                run.g.step([c.data_ptr() for c in run.contribs], which, run.hyper)
            assert run.g.finish(wait=False) is None
            o.step(k)
        st = run.g.step_state()
        assert (st.t, st.scale, st.skipped_total, st.finished) == (o.sc.t, o.sc.scale, 1, 5)
        assert st.good_steps == o.sc.good
        _compare_full(run, o, "enqueued")
    finally:
        run.close()


@pytest.mark.parametrize("staging", [0, 1])
def test_long_run_with_loss_scale_cycles(staging):
    """400 steps enqueued back to back (fp16, 3 buckets, dynamic loss scale growing every 25
    clean steps, one planted inf): t, scale, skip count and every state bit must follow the
    oracle at the end; no drift over hundreds of ping-pong flips and commits."""
    w = _mk(197, _ragged(60, 12, 4000), 5, 2, steps=400, bucket=7_000, dtype=W.FP16,
            scaler=W.Scaler(init_scale=256.0, growth_interval=25), inject=(123, 2, 4_321))
    run = H.Run(w, options={Z.ZERO_OPT_STAGING: staging})
    o = H.OracleFull(w, run.bound)
    try:
        skips = 0
        for k in range(1, w.steps + 1):
            for which, lo, hi in run.ranges():
                for r in range(w.n_d):
                    H.fill_device(run.contribs[r], synth.grad_stream(w, k, r), run.units, lo, hi)
                run.g.step([c.data_ptr() for c in run.contribs], which, run.hyper)
            run.g.finish(wait=False)
            skips += o.step(k)
        st = run.g.step_state()
        assert skips == 1
        assert (st.t, st.scale, st.skipped_total, st.finished, st.good_steps) == \
            (o.sc.t, o.sc.scale, 1, w.steps, o.sc.good)
        _compare_full(run, o, f"after {w.steps} steps")
    finally:
        run.close()


def test_bias_table_saturates():
    """beta1 = 0.5, beta2 = 0.6: 1 - beta^t rounds to 1 after ~72 steps; 90 steps cross the
    end of the table and keep matching the oracle."""
    w = W.Workload(wid=131, name="sat", sizes=tuple(_ragged(14, 8, 3000)), n_d=3, stage=1,
                   bucket_elems=0, unit_first=(), dtype=W.BF16, steps=90,
                   hyper=W.Hyper(beta1=0.5, beta2=0.6), scaler=None)
    run = H.Run(w)
    o = H.OracleFull(w, run.bound)
    try:
        for k in range(1, w.steps + 1):
            res = run.step(k)
            o.step(k)
            assert res.t == k
            if k in (1, 2, 70, 73, 90):
                _compare_full(run, o, f"saturating table, step {k}")
    finally:
        run.close()


@pytest.mark.parametrize("beta2,t0", [(0.999, 40_000), (0.99999, 70_000)])
def test_restored_state_far_into_training(beta2, t0):
    """Resume at t0 applied steps with a non-default loss scale.  With beta2 = 0.99999 the
    bias corrections of t0 + 1 lie beyond the table and are formed on the GPU in double."""
    w = W.Workload(wid=132, name="resume", sizes=tuple(_ragged(15, 10, 5000)), n_d=4, stage=2,
                   bucket_elems=6_000, unit_first=(), dtype=W.FP16, steps=2,
                   hyper=W.Hyper(beta2=beta2), scaler=W.Scaler(init_scale=256.0))
    run = H.Run(w)
    o = H.OracleFull(w, run.bound)
    try:
        state = Z.zero_step_result_t(0, 0, t0, 256.0, 5, 0, t0)
        Z.zero_restore_state(run.g.plan, state)
        o.sc.t, o.sc.good = t0, 5
        for k in (1, 2):
            res = run.step(k)
            o.step(k)
            assert (res.t, res.scale) == (o.sc.t, o.sc.scale)
            _compare_full(run, o, f"restored at t={t0}, step {k}")
    finally:
        run.close()


# ---------------------------------------------------------------------- gradient norm and clipping

def _hyper(max_norm=0.0, report=False):
    return W.Hyper(max_grad_norm=max_norm, report_norm=report)


CLIP_CASES = {
    "z1_nd4_clip": W.Workload(wid=140, name="clip1", sizes=(70_001, 333), n_d=4, stage=1,
                              bucket_elems=0, unit_first=(), dtype=W.BF16, steps=3,
                              hyper=_hyper(0.05), scaler=None),
    "z2_nd8_fp16_buckets_clip_skip": W.Workload(
        wid=141, name="clip2", sizes=tuple(_ragged(16, 40, 9000)), n_d=8, stage=2,
        bucket_elems=10_000, unit_first=(), dtype=W.FP16, steps=4, hyper=_hyper(1e-6),
        scaler=W.Scaler(), outliers=True, inject=(2, 5, 33_333)),
    "z3_nd16_units_clip": W.Workload(
        wid=142, name="clip3", sizes=tuple(_ragged(17, 24, 6000)), n_d=16, stage=3,
        bucket_elems=0, unit_first=(0, 5, 11, 17, 23), dtype=W.BF16, steps=3,
        hyper=_hyper(0.02), scaler=None),
    "z2_nd7_report_only": W.Workload(
        wid=143, name="report", sizes=tuple(_ragged(18, 60, 5000)), n_d=7, stage=2,
        bucket_elems=20_000, unit_first=(), dtype=W.BF16, steps=3, hyper=_hyper(0.0, True),
        scaler=None),
}


def _run_clip(name, options=None):
    w = CLIP_CASES[name]
    run = H.Run(w, options=options)
    o = H.OracleFull(w, run.bound)
    try:
        for k in range(1, w.steps + 1):
            res = run.step(k)
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale
            want = np.sqrt(o.norm2)
            if np.isfinite(want):
                assert abs(res.grad_norm - want) <= 1e-12 * want, (res.grad_norm, want)
            else:
                assert not np.isfinite(res.grad_norm)
            _compare_full(run, o, f"{name} step {k}")
    finally:
        run.close()


@pytest.mark.parametrize("name", list(CLIP_CASES))
def test_norm_and_clipping_full_parity(name):
    _run_clip(name)


def test_report_only_leaves_the_update_unchanged():
    w = CLIP_CASES["z2_nd7_report_only"]
    plain = dataclasses.replace(w, hyper=_hyper(0.0, False))
    a, b = H.Run(w), H.Run(plain)
    try:
        for k in (1, 2):
            ra, rb = a.step(k), b.step(k)
            assert ra.grad_norm > 0 and rb.grad_norm == -1.0
            for r in a.bound:
                x, y = a.read_logical(r), b.read_logical(r)
                for key in x:
                    assert np.array_equal(x[key].view(np.uint32), y[key].view(np.uint32))
    finally:
        a.close()
        b.close()


def test_norm_is_deterministic_and_pass_order_is_checked():
    w = CLIP_CASES["z1_nd4_clip"]
    norms = []
    for _ in range(2):
        run = H.Run(w)
        try:
            norms.append(run.step(1).grad_norm)
        finally:
            run.close()
    assert norms[0] == norms[1]
    run = H.Run(w)
    try:
        ptrs = [c.data_ptr() for c in run.contribs]
        with pytest.raises(Z.ZeroError) as e:            # clipping without the norm pass
            run.g.step(ptrs, -1, run.hyper)
        assert e.value.status == Z.ZERO_ESTATE
        plain = Z.hyper()
        run.g.step(ptrs, -1, plain)
        with pytest.raises(Z.ZeroError) as e:            # the norm must precede the update
            run.g.grad_norm(ptrs, -1)
        assert e.value.status == Z.ZERO_ESTATE
        run.g.finish()
    finally:
        run.close()


# ---------------------------------------------------------------------- overlapped stage-3 schedule

OVERLAP_CASES = {
    "z3_nd16_units": SMALL_CASES["z3_nd16_units"],
    "z3_nd3_fp16_peers_skip_first": SMALL_CASES["z3_nd3_fp16_peers_skip_first"],
    "z3_nd16_units_clip": CLIP_CASES["z3_nd16_units_clip"],
}


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("name", list(OVERLAP_CASES))
def test_overlapped_stage3_schedule_full_parity(name, order):
    """Gathers on a second stream, double-buffered, against the oracle: states, shards and the
    last two gathered units (left in the two buffers) must match.  Units first to last, and
    last to first (ZERO_OPT_UNIT_ORDER = 1)."""
    _run_overlap(OVERLAP_CASES[name], name, options={Z.ZERO_OPT_UNIT_ORDER: order})


def _run_overlap(w, name, options=None):
    order = (options or {}).get(Z.ZERO_OPT_UNIT_ORDER, 0)
    run = H.Run(w, options=options)
    o = H.OracleFull(w, run.bound)
    comm = torch.cuda.Stream()
    nu = len(run.units)
    maxu = int(run.info.max_unit_pad)
    bufs = [torch.empty(max(8, maxu), dtype=torch.int16, device="cuda") for _ in range(2)]
    contribs = [[torch.empty(max(8, U[3]), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
                for U in run.units]
    try:
        for k in range(1, w.steps + 1):
            expect_g = [o.gathered(u) for u in range(nu)]
            for u, (which, lo, hi) in enumerate(run.ranges()):
                for r in range(w.n_d):
                    H.fill_device(contribs[u][r], synth.grad_stream(w, k, r), run.units, lo, hi)
            ptrs = [c.data_ptr() for unit in contribs for c in unit]
            res = Z.zero_step_units_overlapped(run.g.plan, ptrs, [b.data_ptr() for b in bufs],
                                               run.hyper, torch.cuda.current_stream().cuda_stream,
                                               comm.cuda_stream)
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale
            torch.cuda.synchronize()
            seq = list(range(nu))[::-1] if order else list(range(nu))
            for i in range(max(0, nu - 2), nu):            # the last two positions of the order
                u = seq[i]
                got = bufs[i % 2][:run.units[u][3]].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, expect_g[u]), f"gathered unit {u} at step {k}"
            _compare_full(run, o, f"overlapped {name} order {order} step {k}")
    finally:
        run.close()


def test_overlapped_schedule_argument_errors():
    w = SMALL_CASES["z2_nd7_ragged_tensors"]
    run = H.Run(w)
    try:
        s = torch.cuda.current_stream().cuda_stream
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_step_units_overlapped(run.g.plan, [run.contribs[0].data_ptr()] * w.n_d,
                                         [0x1000, 0x2000], run.hyper, s, torch.cuda.Stream().cuda_stream)
        assert e.value.status == Z.ZERO_EINVAL                     # stage 3 only
    finally:
        run.close()


@pytest.mark.parametrize("two_streams", [True, False])
def test_overlapped_schedule_refuses_before_enqueuing(two_streams):
    """A bad argument of any unit (a NULL contribution of the last unit, a unit left gathered, a
    NULL gather buffer, betas out of range) is refused before anything is enqueued: no step is
    left open and no unit gathered, and the next call runs the step the oracle expects."""
    w = dataclasses.replace(SMALL_CASES["z3_nd16_units"], wid=196, steps=1)
    run = H.Run(w)
    o = H.OracleFull(w, run.bound)
    comm = torch.cuda.Stream() if two_streams else None
    nu = len(run.units)
    bufs = [torch.empty(max(8, int(run.info.max_unit_pad)), dtype=torch.int16, device="cuda")
            for _ in range(2)]
    contribs = [[torch.empty(max(8, U[3]), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
                for U in run.units]
    s = torch.cuda.current_stream().cuda_stream
    cs = comm.cuda_stream if comm is not None else None
    try:
        for u, (which, lo, hi) in enumerate(run.ranges()):
            for r in range(w.n_d):
                H.fill_device(contribs[u][r], synth.grad_stream(w, 1, r), run.units, lo, hi)
        ptrs = [c.data_ptr() for unit in contribs for c in unit]
        gptrs = [b.data_ptr() for b in bufs]

        def refused(status, ptrs=ptrs, gptrs=gptrs, hyper=run.hyper):
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_step_units_overlapped(run.g.plan, ptrs, gptrs, hyper, s, cs)
            assert e.value.status == status
            assert not run.g.step_state().t                        # nothing committed
            with pytest.raises(Z.ZeroError) as e:                  # and no step open
                Z.zero_step_finish(run.g.plan, s)
            assert e.value.status == Z.ZERO_ESTATE

        refused(Z.ZERO_EINVAL, ptrs=ptrs[:-1] + [0])               # last unit, last rank
        refused(Z.ZERO_EINVAL, gptrs=[gptrs[0], 0])                # unit 1's buffer
        refused(Z.ZERO_EALIGN, gptrs=[gptrs[0], gptrs[1] + 1])
        refused(Z.ZERO_EINVAL, hyper=Z.hyper(beta1=1.0))
        run.g.gather(nu - 1, bufs[0])
        refused(Z.ZERO_ESTATE)                                     # a unit left gathered
        run.g.release(nu - 1)
        res = Z.zero_step_units_overlapped(run.g.plan, ptrs, gptrs, run.hyper, s, cs)
        flag = o.step(1)
        assert (res.skipped, res.t) == (flag, 1)
        _compare_full(run, o, "overlapped schedule after refused calls")
    finally:
        torch.cuda.synchronize()
        run.close()


# ---------------------------------------------------------------------- FSDP-2 per-parameter plans

def _pp(wid, n_t, n_d, seed, dtype=W.BF16, units=(0,), steps=3, scaler=None, inject=None,
        bound=None, max_rows=300, max_cols=64):
    rng = np.random.default_rng(seed)
    dim0 = [int(x) for x in rng.integers(1, max_rows, size=n_t)]
    sizes = [d * int(c) for d, c in zip(dim0, rng.integers(1, max_cols, size=n_t))]
    return W.Workload(wid=wid, name=f"pp{wid}", sizes=tuple(sizes), n_d=n_d, stage=3,
                      bucket_elems=0, unit_first=tuple(units), dtype=dtype, steps=steps,
                      hyper=W.Hyper(), scaler=scaler, inject=inject, bound_ranks=bound,
                      dim0=tuple(dim0), per_param=True)


PP_CASES = {
    "pp_nd4_units": _pp(150, 20, 4, 1, units=(0, 6, 13)),
    "pp_nd8_fp16_peers_skip": _pp(151, 16, 8, 2, dtype=W.FP16, units=(0, 5, 9),
                                  scaler=W.Scaler(init_scale=512.0), inject=(2, 3, 4_321),
                                  bound=(0, 3, 7)),
    "pp_nd16_rows_below_ranks": _pp(152, 30, 16, 3, units=(0, 10, 20), max_rows=20),
}


@pytest.mark.parametrize("name", list(PP_CASES))
def test_per_param_full_parity(name):
    _run_full(PP_CASES[name])


@pytest.mark.parametrize("mode", ["clip", "clip_offload", "report"])
@pytest.mark.parametrize("name", ["pp_nd4_units", "pp_nd8_fp16_peers_skip"])
def test_per_param_clipping_full_parity(name, mode):
    """FSDP-2 per-parameter plans with the global gradient norm: the norm pre-pass over every
    unit's row chunks, then the clipped updates, on the GPU and offloaded to host threads; or
    the norm reported from the fused pass.  States, shards, skips and the norm against the
    oracle."""
    offload = mode == "clip_offload"
    hyper = _hyper(0.0, True) if mode == "report" else _hyper(1e-3)
    w = dataclasses.replace(PP_CASES[name], wid=PP_CASES[name].wid + 60, hyper=hyper,
                            offload=offload)
    run = H.Run(w)
    o = H.OracleFull(w, run.bound)
    try:
        for k in range(1, w.steps + 1):
            res = run.step(k)
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale, k
            want = np.sqrt(o.norm2)
            if np.isfinite(want):
                assert abs(res.grad_norm - want) <= 1e-12 * want, (res.grad_norm, want)
            else:
                assert not np.isfinite(res.grad_norm)
            mism = _compare_full(run, o, f"per-parameter clip {name} step {k}")
            if offload:
                assert mism == 0
    finally:
        run.close()


@pytest.mark.parametrize("i", [3, 4])
def test_per_param_config_sampled(i):
    w = W.per_param_variant(W.workload(i))
    n, mism = _run_sampled(w, bound=(0, w.n_d - 1) if i == 4 else None)
    print(f"per-parameter {w.name}: {n} sampled elements, {mism} bit mismatches")


@pytest.mark.parametrize("order", [0, 1])
def test_per_param_overlapped_schedule(order):
    _run_overlap(PP_CASES["pp_nd4_units"], "pp", options={Z.ZERO_OPT_UNIT_ORDER: order})


# ---------------------------------------------------------------------- ZeRO-Offload

OFFLOAD_CASES = {
    "z1_nd4": dataclasses.replace(SMALL_CASES["z1_nd4_tiles_ragged_tail"], wid=160, offload=True),
    "z2_nd8_fp16_buckets_inf": dataclasses.replace(SMALL_CASES["z2_nd8_fp16_buckets_inf"], wid=161,
                                                   offload=True),
    "z2_nd5_odd_bucket_scalar_path": dataclasses.replace(
        SMALL_CASES["z2_nd5_odd_bucket_scalar_path"], wid=162, offload=True),
    "z3_nd3_fp16_peers_skip_first": dataclasses.replace(
        SMALL_CASES["z3_nd3_fp16_peers_skip_first"], wid=163, offload=True),
    "pp_nd4_units": dataclasses.replace(PP_CASES["pp_nd4_units"], wid=164, offload=True),
    # several reduction groups (>= 4M elements each) spread over two buckets, fp16 with a
    # skipped second step: the host update of a group starts while later groups and the
    # second bucket are still being reduced, and the flagged step takes the re-cast path
    "z2_nd2_fp16_groups_buckets_skip": dataclasses.replace(
        _mk(165, [9_000_003, 1_700_001], 2, 2, steps=3, bucket=6_000_000, dtype=W.FP16,
            scaler=W.Scaler(), inject=(2, 1, 8_765_431)), offload=True),
}


@pytest.mark.parametrize("name", list(OFFLOAD_CASES))
def test_offload_full_parity(name):
    """Host-CPU AdamW over host-resident state (gradients reduced on the GPU and written to
    pinned host memory) against the oracle: the same fp32 operation order, so 0 mismatches."""
    mism = _run_full(OFFLOAD_CASES[name])
    assert mism == 0


@pytest.mark.parametrize("name", ["z2_nd2_fp16_groups_buckets_skip", "z2_nd8_fp16_buckets_inf",
                                  "z3_nd3_fp16_peers_skip_first", "pp_nd4_units", "z1_nd4"])
def test_offload_deferred_reductions_full_parity(name):
    """ZERO_OPT_OFFLOAD_DEFER: every call runs only its flag pass; the finish, knowing the skip
    decision, streams the reductions (none on a skipped step) while the host threads update.
    Each bucket / unit keeps its own contribution buffers until the finish, as the option
    requires.  Same results as the stream-ordered path: the oracle's, bit for bit."""
    w = OFFLOAD_CASES[name]
    run = H.Run(w, alloc_contribs=False, options={Z.ZERO_OPT_OFFLOAD_DEFER: 1})
    o = H.OracleFull(w, run.bound)
    calls = run.ranges()
    bufs = [[torch.empty(max(8, hi - lo), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
            for (_w, lo, hi) in calls]
    try:
        for k in range(1, w.steps + 1):
            for ci, (which, lo, hi) in enumerate(calls):
                for r in range(w.n_d):
                    H.fill_device(bufs[ci][r], synth.grad_stream(w, k, r), run.units, lo, hi)
                if w.stage == 3:
                    run.g.gather(which, run.gather_buf)
                    run.g.release(which)
                run.g.step([t.data_ptr() for t in bufs[ci]], which, run.hyper)
            res = run.g.finish()
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale, f"step {k}"
            _compare_full(run, o, f"offload deferred {name} step {k}")
    finally:
        run.close()


@pytest.mark.parametrize("defer", [0, 1])
@pytest.mark.parametrize("name", ["z1_nd4_clip", "z2_nd8_fp16_buckets_clip_skip", "z3_nd16_units_clip"])
def test_offload_clipping_full_parity(name, defer):
    """ZeRO-Offload with clipping: the GPU norm pre-pass over every bucket/unit, then the
    reductions to host memory; the host threads scale each gradient by the coefficient formed
    from the step's norm with the GPU's double operations before the update.  Against the
    oracle bit for bit, with the reported norm; stream-ordered and deferred reductions."""
    w = dataclasses.replace(CLIP_CASES[name], wid=CLIP_CASES[name].wid + 50, offload=True)
    run = H.Run(w, alloc_contribs=False, options={Z.ZERO_OPT_OFFLOAD_DEFER: defer})
    o = H.OracleFull(w, run.bound)
    calls = run.ranges()
    # every call keeps its own contribution buffers until the finish (deferred reductions)
    bufs = [[torch.empty(max(8, hi - lo), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
            for (_w, lo, hi) in calls]
    try:
        for k in range(1, w.steps + 1):
            for ci, (which, lo, hi) in enumerate(calls):
                for r in range(w.n_d):
                    H.fill_device(bufs[ci][r], synth.grad_stream(w, k, r), run.units, lo, hi)
                run.g.grad_norm([t.data_ptr() for t in bufs[ci]], which)
            for ci, (which, lo, hi) in enumerate(calls):
                if w.stage == 3:
                    run.g.gather(which, run.gather_buf)
                    run.g.release(which)
                run.g.step([t.data_ptr() for t in bufs[ci]], which, run.hyper)
            res = run.g.finish()
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale, k
            want = np.sqrt(o.norm2)
            if np.isfinite(want):
                assert abs(res.grad_norm - want) <= 1e-12 * want, (res.grad_norm, want)
            else:
                assert not np.isfinite(res.grad_norm)
            assert _compare_full(run, o, f"offload {name} step {k}") == 0
    finally:
        run.close()


def test_offload_worker_threads_end_with_the_plan():
    """An offloaded plan keeps its host worker threads between steps and ends them in
    zero_plan_destroy: the process's thread count returns to where it was."""
    import os
    if not os.path.isdir("/proc/self/task"):
        pytest.skip("needs /proc")
    threads = lambda: len(os.listdir("/proc/self/task"))
    w = OFFLOAD_CASES["z1_nd4"]
    # a first offloaded plan, so that threads the CUDA runtime starts lazily (pinned memory,
    # blocking-sync events, side streams) exist before the count is taken
    warm = H.Run(w)
    try:
        warm.g.offload_threads = 2
        warm.step(1)
    finally:
        warm.close()
    torch.cuda.synchronize()
    before = threads()
    run = H.Run(w)
    try:
        run.g.offload_threads = 6
        for k in (1, 2):
            run.step(k)
        during = threads()
    finally:
        run.close()
    assert during >= before + 6, (before, during)
    assert threads() <= before + 1, (before, threads())   # the pool's six are gone


def test_offload_sampled_config1():
    w = dataclasses.replace(W.workload(1), offload=True)
    n, mism = _run_sampled(w)
    print(f"offloaded {w.name}: {n} sampled elements, {mism} bit mismatches")
    assert mism == 0


def test_offload_rejects_mixing_and_pageable_buffers():
    plan = Z.zero_plan_create([1000], 2, 1, 0, None, Z.ZERO_BF16)
    try:
        n = Z.zero_rank_state_elems(plan, 0)
        ws = torch.zeros(Z.zero_plan_info(plan).workspace_bytes // 4, dtype=torch.int32, device="cuda")
        f16 = torch.zeros(1000, dtype=torch.int16, device="cuda")
        host = [torch.zeros(n, dtype=torch.float32) for _ in range(4)]     # pageable
        p16 = torch.zeros(n, dtype=torch.int16)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_bind_offload(plan, 0, *(h.data_ptr() for h in host), p16.data_ptr(), None,
                                f16.data_ptr(), ws.data_ptr())
        assert e.value.status == Z.ZERO_EINVAL
        dev = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(6)]
        Z.zero_bind(plan, 1, [dev[0].data_ptr(), dev[1].data_ptr()], [dev[2].data_ptr(), dev[3].data_ptr()],
                    [dev[4].data_ptr(), dev[5].data_ptr()], None, f16.data_ptr(), ws.data_ptr())
        pinned = [torch.zeros(n, dtype=torch.float32, pin_memory=True) for _ in range(4)]
        p16p = torch.zeros(n, dtype=torch.int16, pin_memory=True)
        with pytest.raises(Z.ZeroError) as e:                      # on-GPU rank already bound
            Z.zero_bind_offload(plan, 0, *(h.data_ptr() for h in pinned), p16p.data_ptr(), None,
                                f16.data_ptr(), ws.data_ptr())
        assert e.value.status == Z.ZERO_ESTATE
    finally:
        Z.zero_plan_destroy(plan)


# ---------------------------------------------------------------------- tiny-case sweep

def test_tiny_case_sweep():
    """Bounds and peeling: 150 random plans with phi <= 80, N_d 1..16, stages 1/2/3, bf16 and
    fp16, odd buckets, zero-size tensors, and half of them fed contributions that start one
    element past a 16-byte boundary (scalar path); the two step kernels alternate; two steps
    each against the oracle."""
    rng = np.random.default_rng(60)
    for trial in range(150):
        nt = int(rng.integers(1, 7))
        sizes = [int(x) for x in rng.integers(0, 15, size=nt)]
        if sum(sizes) == 0:
            sizes[0] = 1
        n_d = int(rng.integers(1, 17))
        stage = int(rng.integers(1, 4))
        units = ()
        if stage == 3 and nt > 1:
            units = tuple([0] + sorted(set(int(x) for x in rng.integers(1, nt, size=2))))
        bucket = int(rng.integers(0, 30)) if stage == 2 else 0
        dtype = int(rng.integers(0, 2))
        w = W.Workload(wid=300 + trial, name=f"tiny{trial}", sizes=tuple(sizes), n_d=n_d,
                       stage=stage, bucket_elems=bucket, unit_first=units, dtype=dtype, steps=2,
                       hyper=W.Hyper(), scaler=None)
        shift = bool(rng.integers(0, 2))
        run = H.Run(w, options={Z.ZERO_OPT_STAGING: trial % 2})
        o = H.OracleFull(w, run.bound)
        try:
            for k in (1, 2):
                for which, lo, hi in run.ranges():
                    if stage == 3:
                        run.g.gather(which, run.gather_buf)
                        run.g.release(which)
                    ptrs = []
                    for r in range(n_d):
                        H.fill_device(run.contribs[r], synth.grad_stream(w, k, r), run.units, lo, hi)
                        if shift:
                            sh = torch.zeros(run.contribs[r].numel() + 1, dtype=torch.int16, device="cuda")
                            sh[1:] = run.contribs[r]
                            run.contribs[r] = sh[1:]
                        ptrs.append(run.contribs[r].data_ptr())
                    run.g.step(ptrs, which, run.hyper)
                res = run.g.finish()
                flag = o.step(k)
                assert res.skipped == flag == 0 and res.t == k, trial
                _compare_full(run, o, f"tiny case {trial} step {k}")
        finally:
            run.close()


# ---------------------------------------------------------------------- CUDA graph capture

@pytest.mark.parametrize("staging", [0, 1])
@pytest.mark.parametrize("name", ["z2_nd8_fp16_buckets_inf", "z3_nd16_units"])
def test_step_captured_in_a_cuda_graph(name, staging):
    """The step state lives on the device, so a whole step -- every bucket / unit's fused
    launch, the re-cast and the commit -- can be captured once and replayed: replays with new
    gradients written in place into the same buffers must follow the oracle step by step,
    through a skipped step and the loss-scale back-off.  staging 1: the bulk-staged kernel."""
    w = dataclasses.replace(SMALL_CASES[name], steps=5)
    run = H.Run(w, options={Z.ZERO_OPT_STAGING: staging})
    o = H.OracleFull(w, run.bound)
    ranges = run.ranges()
    bufs = [[torch.empty(max(8, hi - lo), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
            for (_, lo, hi) in ranges]

    def fill(k):
        for (which, lo, hi), unit in zip(ranges, bufs):
            for r in range(w.n_d):
                H.fill_device(unit[r], synth.grad_stream(w, k, r), run.units, lo, hi)

    def enqueue():
        for (which, lo, hi), unit in zip(ranges, bufs):
            run.g.step([b.data_ptr() for b in unit], which, run.hyper)
        run.g.finish(wait=False)

    try:
        fill(1)
        enqueue()                              # step 1 uncaptured: builds the bias table
        o.step(1)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        fill(2)
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                enqueue()                      # captured, not run
        skips = 0
        for k in range(2, w.steps + 1):
            if k > 2:
                fill(k)
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            skips += o.step(k)
            st = run.g.step_state()
            assert (st.t, st.scale, st.skipped_total) == (o.sc.t, o.sc.scale, skips)
            _compare_full(run, o, f"graph replay {name} step {k}")
    finally:
        run.close()


# ---------------------------------------------------------------------- the two step kernels
# The cases above run the default choice (the staged kernel where its residency pays off); the
# register-load kernel re-runs them here, and the staged kernel's own tests (forced on) follow.

BULK = {Z.ZERO_OPT_STAGING: Z.ZERO_STAGING_BULK}
LDG = {Z.ZERO_OPT_STAGING: Z.ZERO_STAGING_REGISTER_LOADS}


@pytest.mark.parametrize("n_d,staged", [(2, 0), (6, 1), (7, 1), (8, 1), (12, 0), (16, 1), (20, 1),
                                          (24, 1), (64, 0), (96, 0)])
def test_automatic_kernel_choice(n_d, staged):
    """The default (ZERO_STAGING_AUTO) launches the staged kernel where its ring gives two blocks
    per SM with tiles of 512 elements or more (or three of 512-element tiles) on GB300's 228 KB
    of shared memory per SM, register loads elsewhere; either way the step matches the oracle."""
    w = _mk(180 + n_d, _ragged(40 + n_d, 20, 30000), n_d, 2, steps=1)
    run = H.Run(w)
    o = H.OracleFull(w, run.bound)
    try:
        assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_STAGING) == Z.ZERO_STAGING_AUTO
        assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_LAST_STEP_KERNEL) == -1
        run.step(1)
        o.step(1)
        assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_LAST_STEP_KERNEL) == staged
        _compare_full(run, o, f"automatic choice, N_d = {n_d}")
    finally:
        run.close()


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_register_loads_small_case_full_parity(name):
    _run_full(SMALL_CASES[name], options=LDG)


def test_register_loads_config0_full_parity():
    w = W.workload(0)
    mism = _run_full(w, options=LDG)
    print(f"{w.name}, register loads: {mism} bit mismatches (within tolerance)")


@pytest.mark.parametrize("i", [1, 2, 3, 4])
def test_register_loads_config_sampled(i):
    w = W.workload(i)
    n, mism = _run_sampled(w, bound=(0, w.n_d - 1) if i == 4 else None, options=LDG)
    print(f"{w.name}, register loads: {n} sampled elements, {mism} bit mismatches")


@pytest.mark.parametrize("name", list(CLIP_CASES))
def test_register_loads_norm_and_clipping(name):
    _run_clip(name, options=LDG)


@pytest.mark.parametrize("name", list(PP_CASES))
def test_register_loads_per_param_full_parity(name):
    """Per-parameter plans: one work item per tensor chunk, up to 256 per launch."""
    _run_full(PP_CASES[name], options=LDG)


def test_register_loads_overlapped_schedule():
    _run_overlap(OVERLAP_CASES["z3_nd16_units"], "register loads z3_nd16_units", options=LDG)


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_bulk_staging_small_case_full_parity(name):
    _run_full(SMALL_CASES[name], options=BULK)


@pytest.mark.parametrize("name", list(CLIP_CASES))
def test_bulk_staging_norm_and_clipping(name):
    _run_clip(name, options=BULK)


@pytest.mark.parametrize("name", list(PP_CASES))
def test_bulk_staging_per_param_full_parity(name):
    _run_full(PP_CASES[name], options=BULK)


@pytest.mark.parametrize("name,tile,stages", [
    ("z2_nd7_ragged_tensors", 8, 2), ("z2_nd7_ragged_tensors", 64, 16),
    ("z2_nd8_fp16_buckets_inf", 1024, 3), ("z3_nd16_units", 512, 2),
    ("z1_nd4_tiles_ragged_tail", 4096, 2), ("z1_nd1", 8192, 2)])
def test_bulk_staging_geometries(name, tile, stages):
    """Tiles from one 8-element vector to 8192 elements and rings of 2 to 16 buffers, over
    ragged tensors, buckets and units (segments shorter than a tile, tiles cut at segment
    ends, one tile larger than the whole model)."""
    _run_full(SMALL_CASES[name], options={Z.ZERO_OPT_STAGING: 1, Z.ZERO_OPT_BULK_TILE: tile,
                                          Z.ZERO_OPT_BULK_STAGES: stages})


GATHER_BULK = {Z.ZERO_OPT_GATHER_STAGING: Z.ZERO_STAGING_BULK}
GATHER_LDG = {Z.ZERO_OPT_GATHER_STAGING: Z.ZERO_STAGING_REGISTER_LOADS}
STAGE3_SMALL = [n for n, w in SMALL_CASES.items() if w.stage == 3]


@pytest.mark.parametrize("gather", ["ldg", "bulk"])
@pytest.mark.parametrize("name", STAGE3_SMALL)
def test_gather_kernels_small_stage3_full_parity(name, gather):
    """Both gather kernels (register loads, bulk-staged) on every stage-3 case: each gathered
    unit equals the oracle's concatenation of the rank shards, bit for bit, at every step."""
    _run_full(SMALL_CASES[name], options=GATHER_BULK if gather == "bulk" else GATHER_LDG)


@pytest.mark.parametrize("gather", ["ldg", "bulk"])
@pytest.mark.parametrize("name", list(PP_CASES))
def test_gather_kernels_per_param_full_parity(name, gather):
    """Per-parameter gathers: up to 256 row-block chunks per launch, ragged and tiny."""
    _run_full(PP_CASES[name], options=GATHER_BULK if gather == "bulk" else GATHER_LDG)


@pytest.mark.parametrize("chunk,stages", [(8, 3), (64, 32), (1000, 5), (32768, 3), (4096, 12)])
def test_bulk_gather_geometries(chunk, stages):
    """Bulk-staged gather rings from one 8-element vector per copy to 64 KB copies, 3 to 32
    entries (loads 1 to 30 chunks ahead), on units with shards shorter than a chunk, ragged
    tails and empty tensors."""
    # set in an order whose intermediate ring fits (the default is 4 entries of 16384)
    order = ([Z.ZERO_OPT_GATHER_CHUNK, Z.ZERO_OPT_GATHER_STAGES] if chunk <= 16384
             else [Z.ZERO_OPT_GATHER_STAGES, Z.ZERO_OPT_GATHER_CHUNK])
    value = {Z.ZERO_OPT_GATHER_CHUNK: chunk, Z.ZERO_OPT_GATHER_STAGES: stages}
    options = {Z.ZERO_OPT_GATHER_STAGING: 1, **{k: value[k] for k in order}}
    for name in ("z3_nd16_units", "z3_nd3_fp16_peers_skip_first", "z3_nd16_empty_unit_tensors"):
        _run_full(SMALL_CASES[name], options=options)


@pytest.mark.parametrize("gather", ["ldg", "bulk"])
@pytest.mark.parametrize("i", [3, 4])
def test_gather_kernels_config_sampled(i, gather):
    w = W.workload(i)
    n, mism = _run_sampled(w, bound=(0, w.n_d - 1) if i == 4 else None,
                           options=GATHER_BULK if gather == "bulk" else GATHER_LDG)
    print(f"{w.name}, {gather} gather: {n} sampled elements, {mism} bit mismatches")


@pytest.mark.parametrize("gather", [Z.ZERO_STAGING_AUTO, Z.ZERO_STAGING_BULK])
def test_gather_of_peer_shards_without_a_bound_rank(gather):
    """A stage-3 plan whose ranks are all peers (16-bit shards only, no workspace): the staged
    gather needs the workspace's error word, so the call falls back to register copies; every
    gathered unit is the concatenation of the rank shards' slices, padding included."""
    sizes, n_d, units = [70_001, 5, 123_457, 33, 4_000_003], 4, [0, 2, 4]
    plan = Z.zero_plan_create(sizes, n_d, 3, 0, units)
    try:
        Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_STAGING, gather)
        gen = torch.Generator(device="cpu").manual_seed(7)
        shards = []
        for r in range(n_d):
            n = Z.zero_rank_state_elems(plan, r)
            sh = torch.randint(-32768, 32767, (n,), dtype=torch.int16, generator=gen).cuda()
            Z.zero_bind_peer(plan, r, sh.data_ptr())
            shards.append(sh)
        layout = Z.zero_plan_tables(plan, Z.ZERO_TABLE_STATE_LAYOUT)   # rank, unit, offset, n
        info = Z.zero_plan_info(plan)
        for u in range(int(info.n_units)):
            parts = [(r, off, n) for (r, uu, off, n) in layout if uu == u]
            total = sum(n for _, _, n in parts)
            dst = torch.full((max(8, total),), -1, dtype=torch.int16, device="cuda")
            Z.zero_gather_layer(plan, u, dst.data_ptr())
            Z.zero_release_layer(plan, u)
            want = torch.cat([shards[r][off:off + n] for r, off, n in sorted(parts)])
            torch.cuda.synchronize()
            assert torch.equal(dst[:total], want), f"unit {u}"
    finally:
        Z.zero_plan_destroy(plan)


def test_bulk_gather_wait_limit_runs_out_and_the_step_is_discarded():
    """A gather whose barrier wait runs out (limit 0) records it in the plan's error word,
    drains its copies and returns; the step then finishing reports ZERO_ETIMEOUT and is
    discarded, and the next step (a full wait limit again) follows the oracle."""
    w = _mk(171, [3_000_000 + 5, 2_500_000, 17], 4, 3, steps=2, units=(0, 1))
    run = H.Run(w, options={**GATHER_BULK, **LDG})
    o = H.OracleFull(w, run.bound)
    try:
        res = run.step(1)
        o.step(1)
        assert res.t == 1
        before = {r: run.read_logical(r) for r in run.bound}
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 0)
        with pytest.raises(Z.ZeroError) as e:
            run.step(2)
        assert e.value.status == Z.ZERO_ETIMEOUT
        st = e.value.result
        assert (st.t, st.finished, st.skipped) == (1, 1, 1)
        for r in run.bound:
            now = run.read_logical(r)
            for key in now:
                assert np.array_equal(now[key].view(np.uint32), before[r][key].view(np.uint32)), key
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 1_000_000_000)
        res = run.step(2)
        o.step(2)
        assert (res.t, res.finished, res.skipped) == (2, 2, 0)
        _compare_full(run, o, "after the gather timeout")
    finally:
        run.close()


def test_bulk_staging_is_bit_identical_to_register_loads():
    w = dataclasses.replace(SMALL_CASES["z2_nd8_fp16_buckets_inf"], steps=4)
    a, b = H.Run(w, options=LDG), H.Run(w, options=BULK)
    try:
        for k in range(1, w.steps + 1):
            ra, rb = a.step(k), b.step(k)
            assert (ra.skipped, ra.t, ra.scale) == (rb.skipped, rb.t, rb.scale)
            for r in a.bound:
                x, y = a.read_logical(r), b.read_logical(r)
                for key in x:
                    assert np.array_equal(x[key].view(np.uint32), y[key].view(np.uint32)), (k, r, key)
            assert torch.equal(a.g.full16, b.g.full16), k
    finally:
        a.close()
        b.close()


def test_bulk_staging_first_launch_inside_a_graph_capture():
    """A plan that stepped with register loads switches to the staged kernel, whose first launch
    (kernel attributes, occupancy query) then happens inside a CUDA graph capture; the replays
    must follow the oracle."""
    w = dataclasses.replace(SMALL_CASES["z2_nd7_ragged_tensors"], wid=175, steps=3)
    run = H.Run(w, options=LDG)
    o = H.OracleFull(w, run.bound)
    try:
        res = run.step(1)
        o.step(1)
        assert res.t == 1
        run.g.set_option(Z.ZERO_OPT_STAGING, 1)
        run.g.set_option(Z.ZERO_OPT_BULK_TILE, 72)      # a geometry no other test launches
        ranges = run.ranges()
        bufs = [[torch.empty(max(8, hi - lo), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
                for (_, lo, hi) in ranges]
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for (which, lo, hi), unit in zip(ranges, bufs):
                    run.g.step([b.data_ptr() for b in unit], which, run.hyper)
                run.g.finish(wait=False)
        for k in (2, 3):
            for (which, lo, hi), unit in zip(ranges, bufs):
                for r in range(w.n_d):
                    H.fill_device(unit[r], synth.grad_stream(w, k, r), run.units, lo, hi)
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            o.step(k)
            assert run.g.step_state().t == k
            _compare_full(run, o, f"staged kernel first captured, step {k}")
    finally:
        run.close()


def test_two_plans_step_concurrently_from_two_threads():
    """Two plans (N_d 7 staged, N_d 12 register loads under the automatic choice) stepped at
    the same time from two host threads on two streams: the library's per-kernel caches and
    per-thread error text are shared, the results must still match the oracle."""
    import threading
    cases = [_mk(195, _ragged(50, 25, 20000), 7, 2, steps=3, bucket=30_000),
             _mk(196, _ragged(51, 25, 20000), 12, 2, steps=3)]
    runs = [H.Run(w) for w in cases]
    oracles = [H.OracleFull(w, r.bound) for w, r in zip(cases, runs)]
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for k in range(1, cases[i].steps + 1):
                    runs[i].step(k)
            stream.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    try:
        threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        torch.cuda.synchronize()
        for w, run, o in zip(cases, runs, oracles):
            for k in range(1, w.steps + 1):
                o.step(k)
            assert run.g.step_state().t == w.steps
            _compare_full(run, o, f"concurrent plan N_d = {w.n_d}")
    finally:
        for run in runs:
            run.close()


def test_bulk_staging_wait_limit_runs_out_and_the_step_is_discarded():
    """A wait limit of 0 makes the first barrier wait that is not already satisfied give up:
    the kernel records it, drains its copies and returns; zero_step_finish reports
    ZERO_ETIMEOUT, the step is discarded (state bits, t, scale and counters unchanged, 16-bit
    parameters rewritten from the unchanged master), and the next step runs normally."""
    w = _mk(170, [4_000_000 + 13], 4, 1, steps=2)
    run = H.Run(w, options=BULK)
    o = H.OracleFull(w, run.bound)
    try:
        res = run.step(1)
        o.step(1)
        assert res.t == 1
        _compare_full(run, o, "before the timeout")
        before = {r: run.read_logical(r) for r in run.bound}
        f16 = run.g.full16.clone()
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 0)
        with pytest.raises(Z.ZeroError) as e:
            run.step(2)
        assert e.value.status == Z.ZERO_ETIMEOUT
        st = e.value.result
        assert (st.t, st.finished, st.skipped_total, st.skipped) == (1, 1, 0, 1)
        for r in run.bound:
            now = run.read_logical(r)
            for key in now:
                assert np.array_equal(now[key].view(np.uint32), before[r][key].view(np.uint32)), key
        assert torch.equal(run.g.full16, f16)
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 1_000_000_000)
        st = run.g.step_state()                 # the report cleared the condition
        assert (st.t, st.finished) == (1, 1)
        res = run.step(2)
        o.step(2)
        assert (res.t, res.finished, res.skipped) == (2, 2, 0)
        _compare_full(run, o, "after the timeout")
    finally:
        run.close()
