"""GPU parity of the host-buffer step (zero_step_host / zero_step_host_finish).

Each rank's 16-bit gradient contribution sits in pinned host memory; the library copies the
slices the bound ranks read into a device staging area (the next call's copies running while
this call's step does), runs the fused step, and copies the updated 16-bit parameters back
to host memory.  Compared with the oracle on the same seeded inputs: the device state
element by element, and the host-side 16-bit results against the oracle's parameters;
skipped steps included (their re-cast parameters must reach the host too).

Tolerances as everywhere: fp32 |gpu - oracle| <= 1e-6 |oracle| + 1e-8, 16-bit <= 1 ulp,
skip decisions, t and the loss scale exact, byte counts exact.
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
    Z.lib()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _mk(wid, sizes, n_d, stage, steps=3, bucket=0, units=(), dtype=W.BF16, scaler=None,
        outliers=False, inject=None, bound=None, hyper=None):
    return W.Workload(wid=wid, name=f"host{wid}", sizes=tuple(sizes), n_d=n_d, stage=stage,
                      bucket_elems=bucket, unit_first=tuple(units), dtype=dtype, steps=steps,
                      hyper=hyper or W.Hyper(), scaler=scaler, outliers=outliers, inject=inject,
                      bound_ranks=bound)


def _ragged(seed, n, hi):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1, hi, size=n)]


CASES = {
    # ZeRO-2 buckets, fp16, loss scale, a planted inf at step 2 (skip + back-off)
    "z2_nd8_fp16_buckets_skip": _mk(401, _ragged(2, 40, 9000), 8, 2, steps=4, bucket=10_000,
                                    dtype=W.FP16, scaler=W.Scaler(), outliers=True,
                                    inject=(2, 3, 77_777)),
    # one call over the whole buffer, ragged tiles
    "z1_nd4_one_call": _mk(402, [3 * 65536 + 13], 4, 1),
    # a subset of the ranks bound: only their shard slices are copied
    "z2_nd8_subset_bound": _mk(403, _ragged(9, 25, 8000), 8, 2, bucket=8000, bound=(1, 6)),
    # ZeRO-3 units with peers and a skipped first step
    "z3_nd3_fp16_peers_skip_first": _mk(404, _ragged(5, 12, 3000), 3, 3, units=(0, 4, 9),
                                        dtype=W.FP16, scaler=W.Scaler(init_scale=1024.0),
                                        inject=(1, 2, 1234), bound=(0, 2)),
    "z3_nd16_units": _mk(405, _ragged(4, 24, 6000), 16, 3, units=(0, 5, 11, 17, 23)),
    # odd bucket size: the scalar path of the kernel on the staged contributions
    "z2_nd5_odd_bucket": _mk(406, _ragged(3, 30, 7000), 5, 2, bucket=12_345),
    # the gradient norm reported over the buckets' calls
    "z2_nd4_buckets_norm": _mk(414, _ragged(6, 30, 9000), 4, 2, bucket=30_000,
                               hyper=W.Hyper(report_norm=True)),
}


def _expected_host16(run, o, which, lo, hi):
    """(mask, values) of the host result of call `which` (range [lo, hi)): the oracle's 16-bit
    parameters of the elements the bound ranks own."""
    w = run.w
    n = hi - lo
    mask = np.zeros(n, dtype=bool)
    want = np.zeros(n, dtype=np.uint16)
    if w.per_param:
        for (r, u, _t, _row0, rows, cols, _cr, coff, soff) in o.pp.chunks:
            if u == which and rows and r in run.bound:
                mask[coff:coff + rows * cols] = True
                want[coff:coff + rows * cols] = o.sh16[r][soff:soff + rows * cols]
        return mask, want
    if w.stage == 3:
        (_f, _c, _numel, _pad, S, _base, sb) = o.units[which]
        for r in run.bound:
            mask[r * S:(r + 1) * S] = True
            want[r * S:(r + 1) * S] = o.sh16[r][sb:sb + S]
        return mask, want
    S = o.units[0][4]
    idx = np.arange(lo, hi)
    mask = np.isin(idx // S, run.bound)
    want = o.full16[lo:hi].copy()
    return mask, want


def _run_host(w, pipeline, one_call=False, options=None):
    run = H.Run(w, alloc_contribs=False, options=options)
    o = H.OracleFull(w, run.bound)
    try:
        run.g.bind_host_staging()
        run.g.set_option(Z.ZERO_OPT_HOST_PIPELINE, pipeline)
        calls = run.ranges()
        # one pinned set per call: the copies of one call may still run while the next is filled
        host = [[torch.zeros(max(8, hi - lo), dtype=torch.int16, pin_memory=True)
                 for _ in range(w.n_d)] for (_w, lo, hi) in calls]
        out = [torch.zeros(max(8, hi - lo), dtype=torch.int16, pin_memory=True)
               for (_w, lo, hi) in calls]
        gbuf = run.gather_buf
        clip = w.hyper.max_grad_norm > 0
        for k in range(1, w.steps + 1):
            expect_h2d = expect_d2h = 0
            if clip:                             # every call's norm pre-pass from host memory first
                for ci, (which, lo, hi) in enumerate(calls):
                    for r in range(w.n_d):
                        vals = H.fill_host(synth.grad_stream(w, k, r), run.units, lo, hi)
                        host[ci][r][:hi - lo].copy_(torch.from_numpy(vals.view(np.int16)))
                    run.g.grad_norm_host([t.data_ptr() for t in host[ci]], -1 if one_call else which)
                    mask, _ = _expected_host16(run, o, which, lo, hi)
                    expect_h2d += 2 * w.n_d * int(mask.sum())
            for ci, (which, lo, hi) in enumerate(calls):
                if not clip:
                    for r in range(w.n_d):
                        vals = H.fill_host(synth.grad_stream(w, k, r), run.units, lo, hi)
                        host[ci][r][:hi - lo].copy_(torch.from_numpy(vals.view(np.int16)))
                if w.stage == 3:
                    run.g.gather(which, gbuf)
                    run.g.release(which)
                call = -1 if one_call else which
                run.g.step_host([t.data_ptr() for t in host[ci]], call, run.hyper,
                                out[ci].data_ptr())
                mask, _ = _expected_host16(run, o, which, lo, hi)
                owned = int(mask.sum())
                expect_h2d += 2 * w.n_d * owned   # every contribution's slices of owned elements
                expect_d2h += 2 * owned
            res = run.g.finish_host()
            flag = o.step(k)
            assert res.skipped == flag, f"step {k}"
            assert res.t == o.sc.t and res.scale == o.sc.scale, f"step {k}"
            if w.hyper.report_norm or clip:             # summed over every launch of the step
                # The GPU sums fp32(g*g) per thread as an error-free pair of floats and the
                # block partials in double; the oracle sums them in double in flat order.  Both
                # stay within about n * 2^-53 of the exact sum; over these sizes (<= 34M
                # elements) 1e-10 of the norm bounds the difference.
                want = np.sqrt(o.norm2)
                if np.isfinite(want):
                    assert abs(res.grad_norm - want) <= 1e-10 * want, (k, res.grad_norm, want)
                else:                                    # a non-finite gradient: no norm
                    assert not np.isfinite(res.grad_norm), (k, res.grad_norm)
            H.compare_full(run, o, f"{w.name} host step {k}")
            for ci, (which, lo, hi) in enumerate(calls):
                mask, want = _expected_host16(run, o, which, lo, hi)
                got = out[ci][:hi - lo].numpy().view(np.uint16)
                H.assert_16_close(got[mask], want[mask], f"{w.name} step {k} call {which} host16")
            h2d = Z.zero_get_option(run.g.plan, Z.ZERO_OPT_HOST_H2D_BYTES)
            d2h = Z.zero_get_option(run.g.plan, Z.ZERO_OPT_HOST_D2H_BYTES)
            # a skipped step copies its re-cast parameters once more
            assert d2h == expect_d2h * (2 if flag else 1), (k, d2h, expect_d2h)
            assert h2d == expect_h2d, (k, h2d, expect_h2d)
    finally:
        run.close()


@pytest.mark.parametrize("pipeline", [1, 0])
@pytest.mark.parametrize("name", list(CASES))
def test_host_path_full_parity(name, pipeline):
    _run_host(CASES[name], pipeline)


def test_host_path_tiny_case_sweep():
    """Bounds of the copy lists: 80 random plans with phi <= 120, N_d 1..16, stages 1/2/3, bf16
    and fp16, odd buckets, zero-size tensors and random subsets of the ranks bound, fed from
    host memory pipelined and serial in turn; two steps each against the oracle (device state,
    host results and byte counts)."""
    rng = np.random.default_rng(61)
    for trial in range(80):
        nt = int(rng.integers(1, 7))
        sizes = [int(x) for x in rng.integers(0, 21, size=nt)]
        if sum(sizes) == 0:
            sizes[0] = 1
        n_d = int(rng.integers(1, 17))
        stage = int(rng.integers(1, 4))
        units = ()
        if stage == 3 and nt > 1:
            units = tuple([0] + sorted(set(int(x) for x in rng.integers(1, nt, size=2))))
        bucket = int(rng.integers(0, 40)) if stage == 2 else 0
        bound = None
        if n_d > 1 and rng.integers(0, 2):
            bound = tuple(sorted(set(int(x) for x in rng.integers(0, n_d, size=int(rng.integers(1, n_d))))))
        w = _mk(600 + trial, sizes, n_d, stage, steps=2, bucket=bucket, units=units,
                dtype=int(rng.integers(0, 2)), bound=bound)
        _run_host(w, trial % 2)


def test_host_path_one_call_over_the_whole_buffer():
    _run_host(CASES["z1_nd4_one_call"], 1, one_call=True)


@pytest.mark.parametrize("staging", [0, 1])
def test_host_path_both_step_kernels(staging):
    _run_host(CASES["z3_nd16_units"], 1, options={Z.ZERO_OPT_STAGING: staging})


def test_host_path_per_parameter_plan():
    w = W.Workload(wid=407, name="host_pp", sizes=(12 * 7, 5 * 3, 40 * 9, 2 * 11, 64), n_d=4,
                   stage=3, bucket_elems=0, unit_first=(0, 2, 4), dtype=W.BF16, steps=3,
                   hyper=W.Hyper(), scaler=None, dim0=(12, 5, 40, 2, 8), per_param=True,
                   bound_ranks=(0, 3))
    _run_host(w, 1)


def test_host_path_per_parameter_one_unit_split_into_pieces():
    """A per-parameter plan of one unit (two 4096-row tensors, 33.6M elements, 4 ranks): the
    step's only call is cut into pieces whose cuts fall inside the ranks' row chunks."""
    w = W.Workload(wid=418, name="host_pp_pieces", sizes=(4096 * 4096, 4096 * 4100), n_d=4,
                   stage=3, bucket_elems=0, unit_first=(0,), dtype=W.BF16, steps=2,
                   hyper=W.Hyper(), scaler=None, dim0=(4096, 4096), per_param=True)
    _run_host(w, 1)


CLIP_CASES = {
    # clipped steps fed from host memory: the norm pre-pass of every call, then the steps
    "z2_nd8_fp16_buckets_clip_skip": _mk(415, _ragged(16, 40, 9000), 8, 2, steps=4, bucket=10_000,
                                         dtype=W.FP16, scaler=W.Scaler(), outliers=True,
                                         inject=(2, 5, 33_333), hyper=W.Hyper(max_grad_norm=1e-6)),
    "z3_nd16_units_clip": _mk(416, _ragged(17, 24, 6000), 16, 3, units=(0, 5, 11, 17, 23),
                              hyper=W.Hyper(max_grad_norm=0.02)),
    "z1_nd4_two_pieces_clip": _mk(417, [17_000_001, 16_777_259], 4, 1, steps=2,
                                  hyper=W.Hyper(max_grad_norm=0.05)),
    # a per-parameter plan (dim-0 row chunks), two ranks bound
    "pp_nd4_clip": W.Workload(wid=419, name="host_pp_clip", sizes=(12 * 7, 5 * 3, 40 * 9, 2 * 11, 64),
                              n_d=4, stage=3, bucket_elems=0, unit_first=(0, 2, 4), dtype=W.BF16,
                              steps=3, hyper=W.Hyper(max_grad_norm=1e-3), scaler=None,
                              dim0=(12, 5, 40, 2, 8), per_param=True, bound_ranks=(0, 3)),
}


@pytest.mark.parametrize("pipeline", [1, 0])
@pytest.mark.parametrize("name", list(CLIP_CASES))
def test_host_path_clipping_full_parity(name, pipeline):
    """zero_grad_norm_host over every call, then the clipped zero_step_host calls: states,
    host results, the reported norm and the byte counts (the gradients cross the link twice)."""
    _run_host(CLIP_CASES[name], pipeline)


SPLIT_CASES = {
    # one call of 33.8M elements: cut into 2 pieces (a piece is at least 2^24 elements)
    "z1_nd4_two_pieces": _mk(409, [17_000_001, 16_777_259, 777], 4, 1),
    # one fp16 bucket of 50.4M elements over 3 ranks, 2 of them bound: 3 pieces, the cuts
    # inside a rank's shard and across the unbound rank's; an inf at step 2 is skipped
    "z2_nd3_fp16_three_pieces_skip": _mk(410, [25_165_837, 25_165_831, 100_003], 3, 2,
                                         dtype=W.FP16, scaler=W.Scaler(), inject=(2, 1, 8_000_001),
                                         bound=(0, 2)),
    # one ZeRO-3 unit of 33.6M elements over 5 ranks: the call's range is the 5 shards
    "z3_nd5_one_unit_two_pieces": _mk(411, [33_554_467], 5, 3, units=(0,)),
    # the gradient norm reported over the two pieces' launches
    "z1_nd6_two_pieces_norm": _mk(413, [16_800_001, 16_777_259], 6, 1, steps=2,
                                  hyper=W.Hyper(report_norm=True)),
}


@pytest.mark.parametrize("name", list(SPLIT_CASES))
def test_host_path_one_large_call_split_into_pieces(name):
    """A host-buffer call that is the step's only call is cut into pieces of its range, each
    piece's step launch and copy back running while the next piece is copied in; the results
    and the byte counts are those of one call."""
    _run_host(SPLIT_CASES[name], 1)


def test_host_path_bucket_minus_one_split_into_pieces():
    """Bucket -1 on a plan of four buckets: the one call covers every bucket, and its pieces cut
    across bucket, shard and tensor boundaries alike.  Staging areas of the minimum size hold
    one bucket per rank: the call is refused with ZERO_ERANGE and nothing runs; areas of
    N_d * 2 * phi_pad bytes (phi_pad rounded up to 8) take it."""
    w = _mk(412, [12_000_011, 11_999_993, 8_388_608, 1_234_567], 4, 2, steps=2, bucket=9_000_000)
    run = H.Run(w, alloc_contribs=False)
    o = H.OracleFull(w, run.bound)
    try:
        assert len(run.ranges()) == 4
        n = int(run.info.phi_pad)
        host = [torch.zeros(n, dtype=torch.int16, pin_memory=True) for _ in range(w.n_d)]
        out = torch.zeros(n, dtype=torch.int16, pin_memory=True)
        run.g.bind_host_staging()
        with pytest.raises(Z.ZeroError) as e:
            run.g.step_host([t.data_ptr() for t in host], -1, run.hyper, out.data_ptr())
        assert e.value.status == Z.ZERO_ERANGE
        part = 2 * ((n + 7) // 8 * 8)                 # a rank's part: the range, whole 16 bytes
        big = [torch.empty(w.n_d * part, dtype=torch.uint8, device="cuda") for _ in range(2)]
        with pytest.raises(Z.ZeroError) as e:         # 16 bytes short of the rank parts
            Z.zero_bind_host_staging(run.g.plan, [t.data_ptr() for t in big], w.n_d * part - 16)
            run.g.step_host([t.data_ptr() for t in host], -1, run.hyper, out.data_ptr())
        assert e.value.status == Z.ZERO_ERANGE
        Z.zero_bind_host_staging(run.g.plan, [t.data_ptr() for t in big], w.n_d * part)
        for k in range(1, w.steps + 1):
            for r in range(w.n_d):
                vals = H.fill_host(synth.grad_stream(w, k, r), run.units, 0, n)
                host[r].copy_(torch.from_numpy(vals.view(np.int16)))
            run.g.step_host([t.data_ptr() for t in host], -1, run.hyper, out.data_ptr())
            res = run.g.finish_host()
            flag = o.step(k)
            assert (res.skipped, res.t) == (flag, o.sc.t), f"step {k}"
            H.compare_full(run, o, f"bucket -1 host step {k}")
            H.assert_16_close(out.numpy().view(np.uint16), o.full16, f"bucket -1 host step {k} host16")
            assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_HOST_H2D_BYTES) == 2 * w.n_d * n
            assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_HOST_D2H_BYTES) == 2 * n
    finally:
        run.close()


def test_host_path_config2_pipelined_sampled():
    """The bucketed ZeRO-2 GPT-2-small workload at full size (fp16, 5 buckets of 25M, 8 ranks,
    loss scale 2^16) fed from host memory with the bucket copies pipelined, over its first four
    steps (the planted inf at step 3 is skipped); sampled elements against the oracle."""
    w = dataclasses.replace(W.workload(2), steps=4)
    run = H.Run(w, alloc_contribs=False)
    try:
        run.g.bind_host_staging()
        assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_HOST_PIPELINE) == 1
        idx = H.sample_indices(run, 20000)
        o = H.OracleSampled(w, idx)
        calls = run.ranges()
        assert len(calls) == 5
        host = [[torch.empty(hi - lo, dtype=torch.int16, pin_memory=True) for _ in range(w.n_d)]
                for (_w, lo, hi) in calls]
        out = [torch.zeros(hi - lo, dtype=torch.int16, pin_memory=True) for (_w, lo, hi) in calls]
        for k in range(1, w.steps + 1):
            for ci, (which, lo, hi) in enumerate(calls):
                for r in range(w.n_d):
                    synth.grad_stream(w, k, r).host_into(host[ci][r].numpy().view(np.uint16), lo)
                run.g.step_host([t.data_ptr() for t in host[ci]], which, run.hyper,
                                out[ci].data_ptr())
            res = run.g.finish_host()
            flag = o.step(k)
            assert res.skipped == flag and res.t == o.sc.t and res.scale == o.sc.scale, f"step {k}"
            st, g16 = run.read_sampled(idx)
            for key, want in (("master", o.p), ("m", o.m), ("v", o.v)):
                H.assert_state_close(st[key], want, f"config2 host step {k} {key}")
            H.assert_16_close(g16, o.out16, f"config2 host step {k} device 16-bit")
            host16 = np.concatenate([t.numpy().view(np.uint16) for t in out])
            H.assert_16_close(host16[idx], o.out16, f"config2 host step {k} host 16-bit")
            assert Z.zero_get_option(run.g.plan, Z.ZERO_OPT_HOST_H2D_BYTES) == 2 * w.n_d * w.phi
    finally:
        run.close()


def test_host_path_errors():
    w = CASES["z2_nd5_odd_bucket"]
    run = H.Run(w, alloc_contribs=False)
    try:
        plan = run.g.plan
        info = run.info
        calls = run.ranges()
        which, lo, hi = calls[0]
        host = [torch.zeros(hi - lo, dtype=torch.int16, pin_memory=True) for _ in range(w.n_d)]
        out = torch.zeros(hi - lo, dtype=torch.int16, pin_memory=True)
        ptrs = [t.data_ptr() for t in host]
        with pytest.raises(Z.ZeroError) as e:                    # no staging bound
            Z.zero_step_host(plan, ptrs, which, run.hyper, out.data_ptr())
        assert e.value.status == Z.ZERO_ESTATE
        a = torch.empty(int(info.host_staging_bytes) + 64, dtype=torch.uint8, device="cuda")
        with pytest.raises(Z.ZeroError) as e:                    # too small
            Z.zero_bind_host_staging(plan, [a.data_ptr(), a.data_ptr() + 16], int(info.host_staging_bytes) - 2)
        assert e.value.status == Z.ZERO_ERANGE
        with pytest.raises(Z.ZeroError) as e:                    # the two areas overlap
            Z.zero_bind_host_staging(plan, [a.data_ptr(), a.data_ptr() + 16], int(info.host_staging_bytes))
        assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:                    # host memory is not device memory
            Z.zero_bind_host_staging(plan, [host[0].data_ptr(), host[1].data_ptr()], int(info.host_staging_bytes))
        assert e.value.status == Z.ZERO_EINVAL
        run.g.bind_host_staging()
        pageable = np.zeros(hi - lo, dtype=np.uint16)
        with pytest.raises(Z.ZeroError) as e:                    # contributions must be pinned
            Z.zero_step_host(plan, [pageable.ctypes.data] + ptrs[1:], which, run.hyper, out.data_ptr())
        assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:                    # so must the result buffer
            Z.zero_step_host(plan, ptrs, which, run.hyper, pageable.ctypes.data)
        assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:                    # no clipping on this path
            Z.zero_step_host(plan, ptrs, which, Z.hyper(max_grad_norm=1.0), out.data_ptr())
        assert e.value.status in (Z.ZERO_EINVAL, Z.ZERO_ESTATE)
        # a step with host calls must end with zero_step_host_finish (the host buffers stay
        # alive until it returns)
        keep = []
        for (wh, lo2, hi2) in calls:
            hb = [torch.zeros(hi2 - lo2, dtype=torch.int16, pin_memory=True) for _ in range(w.n_d)]
            ob = torch.zeros(hi2 - lo2, dtype=torch.int16, pin_memory=True)
            keep.append((hb, ob))
            Z.zero_step_host(plan, [t.data_ptr() for t in hb], wh, run.hyper, ob.data_ptr())
            with pytest.raises(Z.ZeroError) as e:                # the same bucket twice
                Z.zero_step_host(plan, [t.data_ptr() for t in hb], wh, run.hyper, ob.data_ptr())
            assert e.value.status == Z.ZERO_ESTATE
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_step_finish(plan, torch.cuda.current_stream().cuda_stream)
        assert e.value.status == Z.ZERO_ESTATE
        res = run.g.finish_host()
        assert res.t == 1 and res.skipped == 0
    finally:
        torch.cuda.synchronize()
        run.close()


def test_host_norm_pass_errors():
    w = CASES["z2_nd5_odd_bucket"]
    run = H.Run(w, alloc_contribs=False)
    try:
        plan = run.g.plan
        which, lo, hi = run.ranges()[0]
        host = [torch.zeros(hi - lo, dtype=torch.int16, pin_memory=True) for _ in range(w.n_d)]
        out = torch.zeros(hi - lo, dtype=torch.int16, pin_memory=True)
        ptrs = [t.data_ptr() for t in host]
        with pytest.raises(Z.ZeroError) as e:                    # no staging bound
            Z.zero_grad_norm_host(plan, ptrs, which)
        assert e.value.status == Z.ZERO_ESTATE
        run.g.bind_host_staging()
        pageable = np.zeros(hi - lo, dtype=np.uint16)
        with pytest.raises(Z.ZeroError) as e:                    # contributions must be pinned
            Z.zero_grad_norm_host(plan, [pageable.ctypes.data] + ptrs[1:], which)
        assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:                    # one pointer per rank
            Z.zero_grad_norm_host(plan, ptrs[1:], which)
        assert e.value.status == Z.ZERO_EINVAL
        Z.zero_grad_norm_host(plan, ptrs, which)
        with pytest.raises(Z.ZeroError) as e:                    # the same bucket twice
            Z.zero_grad_norm_host(plan, ptrs, which)
        assert e.value.status == Z.ZERO_ESTATE
        clip = Z.hyper(max_grad_norm=1.0)
        with pytest.raises(Z.ZeroError) as e:                    # clipping needs every bucket's norm
            Z.zero_step_host(plan, ptrs, which, clip, out.data_ptr())
        assert e.value.status == Z.ZERO_ESTATE
        Z.zero_step_host(plan, ptrs, which, Z.hyper(), out.data_ptr())
        with pytest.raises(Z.ZeroError) as e:                    # the norm must precede the steps
            Z.zero_grad_norm_host(plan, ptrs, run.ranges()[1][0])
        assert e.value.status == Z.ZERO_ESTATE
    finally:
        torch.cuda.synchronize()
        run.close()


@pytest.mark.parametrize("base", ["z2_nd8_fp16_buckets_skip", "z1_nd4_two_pieces"])
def test_host_path_discarded_step_copies_the_recast_parameters(base):
    """A barrier wait of the staged kernel that runs out (limit 0) discards the step: the
    finish reports ZERO_ETIMEOUT, the state is unchanged, and the 16-bit parameters re-cast from
    the unchanged master are copied to the host buffers again (the rejected update's values,
    copied after the step, are overwritten).  The next step follows the oracle.  Four buckets
    (four calls), and one call cut into two pieces."""
    w = dataclasses.replace({**CASES, **SPLIT_CASES}[base], wid=408, inject=None, steps=2)
    run = H.Run(w, alloc_contribs=False, options={Z.ZERO_OPT_STAGING: Z.ZERO_STAGING_BULK})
    o = H.OracleFull(w, run.bound)
    try:
        run.g.bind_host_staging()
        calls = run.ranges()
        host = [[torch.zeros(hi - lo, dtype=torch.int16, pin_memory=True) for _ in range(w.n_d)]
                for (_w, lo, hi) in calls]
        out = [torch.zeros(hi - lo, dtype=torch.int16, pin_memory=True) for (_w, lo, hi) in calls]

        def step(k):
            for ci, (which, lo, hi) in enumerate(calls):
                for r in range(w.n_d):
                    vals = H.fill_host(synth.grad_stream(w, k, r), run.units, lo, hi)
                    host[ci][r].copy_(torch.from_numpy(vals.view(np.int16)))
                run.g.step_host([t.data_ptr() for t in host[ci]], which, run.hyper, out[ci].data_ptr())
            return run.g.finish_host()

        res = step(1)
        o.step(1)
        assert res.t == 1
        before = {r: run.read_logical(r) for r in run.bound}
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 0)
        with pytest.raises(Z.ZeroError) as e:
            step(2)
        assert e.value.status == Z.ZERO_ETIMEOUT
        assert e.value.result.t == 1
        for r in run.bound:
            now = run.read_logical(r)
            for key in now:
                assert np.array_equal(now[key].view(np.uint32), before[r][key].view(np.uint32)), key
        # the host holds the parameters of the state after step 1 (the oracle's)
        for ci, (which, lo, hi) in enumerate(calls):
            H.assert_16_close(out[ci].numpy().view(np.uint16), o.full16[lo:hi], f"after the discard, call {which}")
        run.g.set_option(Z.ZERO_OPT_WAIT_LIMIT_NS, 1_000_000_000)
        res = step(2)
        o.step(2)
        assert (res.t, res.skipped) == (2, 0)
        H.compare_full(run, o, "host path after the discarded step")
        for ci, (which, lo, hi) in enumerate(calls):
            H.assert_16_close(out[ci].numpy().view(np.uint16), o.full16[lo:hi], f"step 2, call {which}")
    finally:
        run.close()
