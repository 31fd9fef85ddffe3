"""The no-allocation entry point, checked against the plan-based step and the oracle on the GPU.

Some callers cannot allocate device memory: their host framework has reserved the GPU's
memory for its own pool, or their loop cannot afford cudaMalloc/cudaFree, which may
synchronise the whole device.  Those callers cannot hand zero_bind a workspace, so they use
zero_step_range_noalloc, whose only scratch (the non-finite flag) lives in a static device
array inside the library.  These tests run it through the C ABI and compare it, two steps in
a row, with the plan-based zero_step / zero_step_finish on the same inputs and with the CPU
oracle's step on the same seeded values, within the tolerances the other parity tests use.
This file is collected last on purpose.
"""
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


def _workload(dtype, scaler=None, inject=None):
    # ragged: shard size 91,389 is odd, so ranks 1..3 start off the 16-byte grid
    return W.Workload(wid=300 + dtype, name="noalloc", sizes=(300_001, 17, 65_536), n_d=4, stage=1,
                      bucket_elems=0, unit_first=(), dtype=dtype, steps=2, hyper=W.Hyper(),
                      scaler=scaler, inject=inject)


@pytest.mark.parametrize("dtype", [W.BF16, W.FP16])
def test_noalloc_matches_plan_step_two_calls(dtype):
    w = _workload(dtype, scaler=W.Scaler(init_scale=512.0) if dtype == W.FP16 else None)
    run = H.Run(w)
    o = H.OracleFull(w, run.bound)          # the oracle on the same seeded inputs
    try:
        S = run.units[0][4]
        scale = run.scaler.scale if run.scaler is not None else 1.0
        # the no-alloc side keeps its own copies of every rank's state, in logical order
        mine = {}
        for r in range(w.n_d):
            st = {k: run.g.logical(r, run.g.state_tensor(r, k)).clone() for k in ("master", "m", "v")}
            mine[r] = st
        for k in (1, 2):
            res = run.step(k)                       # the existing entry point (plan-based)
            assert res.skipped == 0
            assert o.step(k) == 0
            # this step's contributions (regenerated into the buffers run.step used)
            for rr in range(w.n_d):
                H.fill_device(run.contribs[rr], synth.grad_stream(w, k, rr), run.units, 0,
                              int(run.info.phi_pad))
            for r in range(w.n_d):
                outs = {key: torch.empty(S, dtype=torch.float32, device="cuda") for key in mine[r]}
                out16 = torch.empty(S, dtype=torch.int16, device="cuda")
                ptrs = [c.data_ptr() + 2 * r * S for c in run.contribs]
                flag = Z.zero_step_range_noalloc(
                    ptrs, S, dtype, mine[r]["master"].data_ptr(), mine[r]["m"].data_ptr(),
                    mine[r]["v"].data_ptr(), outs["master"].data_ptr(), outs["m"].data_ptr(),
                    outs["v"].data_ptr(), out16.data_ptr(), run.hyper, k, scale)
                assert flag == 0
                want = run.read_logical(r)
                for key in ("master", "m", "v"):
                    H.assert_state_close(outs[key].cpu().numpy(), want[key], f"step {k} rank {r} {key}")
                full16 = run.g.full16[r * S:(r + 1) * S].cpu().numpy().view(np.uint16)
                H.assert_16_close(out16.cpu().numpy().view(np.uint16), full16, f"step {k} rank {r} 16-bit")
                # and directly against the oracle
                for key, want in (("master", o.p[r]), ("m", o.m[r]), ("v", o.v[r])):
                    H.assert_state_close(outs[key].cpu().numpy(), want, f"oracle step {k} rank {r} {key}")
                H.assert_16_close(out16.cpu().numpy().view(np.uint16), o.full16[r * S:(r + 1) * S],
                                  f"oracle step {k} rank {r} 16-bit")
                mine[r] = outs                      # the next call reads this call's outputs
    finally:
        run.close()


def test_noalloc_flag_and_limits():
    n, n_d = 1000, 3
    contribs = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(n_d)]
    contribs[1][777] = 0x7F80                       # +inf in bf16
    st = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(6)]
    out16 = torch.empty(n, dtype=torch.int16, device="cuda")
    args = [st[0].data_ptr(), st[1].data_ptr(), st[2].data_ptr(), st[3].data_ptr(),
            st[4].data_ptr(), st[5].data_ptr(), out16.data_ptr()]
    assert Z.zero_step_range_noalloc([c.data_ptr() for c in contribs], n, Z.ZERO_BF16, *args,
                                     Z.hyper(), 1) == 1
    contribs[1][777] = 0                            # the flag is cleared at the start of each call
    assert Z.zero_step_range_noalloc([c.data_ptr() for c in contribs], n, Z.ZERO_BF16, *args,
                                     Z.hyper(), 1) == 0
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_step_range_noalloc([contribs[0].data_ptr()] * (Z.ZERO_MAX_RANKS + 1), n,
                                  Z.ZERO_BF16, *args, Z.hyper(), 1)
    assert e.value.status == Z.ZERO_ERANGE
    with pytest.raises(Z.ZeroError) as e:           # output aliasing its input
        Z.zero_step_range_noalloc([c.data_ptr() for c in contribs], n, Z.ZERO_BF16, args[0],
                                  args[1], args[2], args[0], args[4], args[5], args[6], Z.hyper(), 1)
    assert e.value.status == Z.ZERO_EINVAL
