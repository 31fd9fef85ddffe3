"""GPU parity of the launch sequence bench.py times, at the bench's default workload size.

The ZeRO-3 1.3B GPT workload (N_d = 16, 26 units) is bound through the bench's own Bench class,
with its contribution sets and its one-stream schedule (unit 0 gathered by a launch of its own,
then every unit's step launch also gathering the next unit).  Step 1 runs eagerly, as the
bench's warm-up does; step 2 is captured as a CUDA graph on a side stream and replayed twice,
as the timed region is.  After every step, sampled elements (20k random plus every shard,
unit, tensor and padding edge +-9) are compared with the oracle: the fp32 state within
1e-6 |x| + 1e-8, the 16-bit shards within 1 ulp, t and the skip decision exactly; and the last
two units gathered (left in the bench's two gather buffers) bit for bit at sampled positions:
each was gathered inside the previous unit's step launch, from its shards as they were before
this step updated them.
"""
import numpy as np
import pytest
import torch

import bench
import gpu_harness as H
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


def test_bench_default_schedule_graph_replay_sampled():
    w = W.workload(bench.DEFAULT_CONFIG)
    assert w.stage == 3
    b = bench.Bench(w, mem_budget_gb=90.0, n_sets_wanted=2,
                    options={Z.ZERO_OPT_STAGING: Z.ZERO_STAGING_AUTO}, fused_gather=True)
    try:
        assert b.n_sets == 2 and b.all_bound
        idx = H.sample_indices(b.run, 20000)
        o = H.OracleSampled(w, idx)
        nu = len(b.calls)
        rng = np.random.default_rng(1)
        # the last two units at sampled positions: flat index = unit base + position
        gpos, og = {}, {}
        for u in (nu - 2, nu - 1):
            n = int(b.units[u][3])
            gpos[u] = np.unique(np.concatenate([np.arange(min(64, n)), np.arange(max(0, n - 64), n),
                                                rng.integers(0, n, size=4096)])).astype(np.int64)
            og[u] = H.OracleSampled(w, int(b.units[u][5]) + gpos[u])

        def step_and_check(k, t, grads, run_step):
            before = {u: og[u].out16.copy() for u in og}
            run_step()
            torch.cuda.synchronize()
            flag = o.step(grads)
            for u in og:
                og[u].step(grads)
            st, g16 = b.run.read_sampled(idx)
            for key, want in (("master", o.p), ("m", o.m), ("v", o.v)):
                H.assert_state_close(st[key], want, f"bench path step {k} {key}")
            H.assert_16_close(g16, o.out16, f"bench path step {k} shard16")
            state = b.g.step_state()
            assert (state.t, state.skipped) == (t, flag), k
            for u in og:
                buf = b.gather_bufs()[u % 2]
                got = buf[torch.from_numpy(gpos[u]).cuda()].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, before[u]), f"step {k}: unit {u} gathered"

        # step 1, eagerly (contribution set s holds the gradients of step s + 1)
        step_and_check(1, 1, 1, lambda: b.step(b.sets[0]))
        assert b.gather_in_step is True
        # step 2's launches (set 1), captured once and replayed twice like the timed region
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                b.step(b.sets[1])
        torch.cuda.synchronize()
        for k in (2, 3):
            step_and_check(k, k, 2, graph.replay)
    finally:
        torch.cuda.synchronize()
        b.run.close()
