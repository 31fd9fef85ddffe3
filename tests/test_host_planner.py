"""Host-side checks of libzero (no GPU): exports, tables vs the oracle, accounting, errors."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import zero_sharded_mixed_03_gb300 as Z
from synth import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_symbol():
    with open(os.path.join(ROOT, "include", "zero.h")) as f:
        text = f.read()
    declared = set(re.findall(r"^\s*(?:zero_status_t|const char\*|void)\s+(zero_\w+)\s*\(", text, re.M))
    assert len(declared) >= 15
    L = Z.lib()
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert declared <= set(Z.EXPORTED)


def test_binding_constants_match_the_header():
    """Every ZERO_* constant of include/zero.h (enums and #defines) has the same value in the
    Python binding."""
    with open(os.path.join(ROOT, "include", "zero.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    values = {}
    for body in re.findall(r"enum\s*(?:\w+\s*)?\{(.*?)\}", text, re.S):
        nxt = 0
        for item in body.split(","):
            item = item.strip()
            if not item:
                continue
            name, _, val = item.partition("=")
            name = name.strip()
            nxt = int(val.strip(), 0) if val.strip() else nxt
            values[name] = nxt
            nxt += 1
    for name, val in re.findall(r"#define\s+(ZERO_\w+)\s+(\d+)", text):
        values[name] = int(val)
    assert len(values) >= 25
    for name, val in sorted(values.items()):
        if hasattr(Z, name):
            assert getattr(Z, name) == val, name
    missing = [n for n in values if n.startswith("ZERO_OPT_") and not hasattr(Z, n)]
    assert not missing, missing


def _plan_for(sizes, n_d, stage, bucket=0, units=None, dtype=Z.ZERO_BF16):
    return Z.zero_plan_create(list(sizes), n_d, stage, bucket, list(units) if units else None, dtype)


def _compare_tables(sizes, n_d, stage, bucket, units):
    plan = _plan_for(sizes, n_d, stage, bucket, units)
    try:
        L = oracle.Layout(sizes, n_d, units)
        assert [r[0] for r in Z.zero_plan_tables(plan, Z.ZERO_TABLE_TENSOR_OFFSET)] == \
            [int(x) for x in L.tensor_offset]
        assert Z.zero_plan_tables(plan, Z.ZERO_TABLE_UNITS) == [tuple(int(x) for x in u) for u in L.units]
        assert Z.zero_plan_tables(plan, Z.ZERO_TABLE_SHARD_SEGMENTS) == \
            [tuple(int(x) for x in r) for r in L.shard_segments()]
        if stage != 3:
            assert Z.zero_plan_tables(plan, Z.ZERO_TABLE_BUCKET_SEGMENTS) == \
                [tuple(int(x) for x in r) for r in L.bucket_segments(bucket)]
        info = Z.zero_plan_info(plan)
        assert info.phi == sum(sizes) and info.phi_pad == L.total_pad and info.shard == L.shard_total
        # accounting == oracle closed forms
        mem = Z.zero_memory_report(plan)
        om = oracle.memory(L.total_pad, n_d)
        assert [mem.logical[s][c] for s in range(4) for c in range(3)] == [int(x) for x in om[:12]]
        assert mem.logical_ddp_fp32_grads == int(om[12])
        com = Z.zero_comm_report(plan)
        oc = oracle.comm(L.total_pad, n_d)
        assert [com.ddp, com.zero1, com.zero2, com.zero3] == [int(x) for x in oc]
        assert com.this_stage == int(oc[stage])
        _check_state_layout(plan, L, n_d)
    finally:
        Z.zero_plan_destroy(plan)


def _check_state_layout(plan, L, n_d):
    rows = Z.zero_plan_tables(plan, Z.ZERO_TABLE_STATE_LAYOUT)
    assert len(rows) == n_d * len(L.units)
    for r in range(n_d):
        elems = Z.zero_rank_state_elems(plan, r)
        mine = [row for row in rows if row[0] == r]
        end = 0
        for (rr, u, off, n), U in zip(mine, L.units):
            assert n == U[4]
            assert off >= end                           # no overlap, unit order kept
            assert (off - r * n) % 8 == 0               # phase of the 16-bit shard start
            assert off - end < 8                        # gap below one vector
            end = off + n
        assert end <= elems and elems % 8 == 0 and elems - end < 8


def test_tables_match_oracle_random():
    rng = np.random.default_rng(20)
    for _ in range(300):
        nt = int(rng.integers(0, 14))
        sizes = [int(x) for x in rng.integers(0, 40, size=nt)]
        n_d = int(rng.integers(1, 17))
        stage = int(rng.integers(1, 4))
        units, bucket = None, 0
        if stage == 3 and nt > 1 and rng.random() < 0.7:
            cuts = sorted(set(int(x) for x in rng.integers(1, nt, size=int(rng.integers(1, 4)))))
            units = [0] + cuts
        if stage != 3:
            bucket = int(rng.integers(0, 50))
        _compare_tables(sizes, n_d, stage, bucket, units)


@pytest.mark.parametrize("i", range(W.N_WORKLOADS))
def test_tables_match_oracle_workloads(i):
    w = W.workload(i)
    _compare_tables(w.sizes, w.n_d, w.stage, w.bucket_elems, w.unit_first or None)


def test_workload_shapes_in_planner():
    # GPT-2, 1.3B and Llama shapes: all shards a multiple of 8 elements (vector phase 0 everywhere)
    for i in (2, 3, 4):
        w = W.workload(i)
        plan = _plan_for(w.sizes, w.n_d, w.stage, w.bucket_elems, w.unit_first or None)
        rows = Z.zero_plan_tables(plan, Z.ZERO_TABLE_UNITS)
        assert all(u[4] % 8 == 0 for u in rows)
        Z.zero_plan_destroy(plan)
    w = W.workload(2)
    plan = _plan_for(w.sizes, w.n_d, w.stage, w.bucket_elems)
    info = Z.zero_plan_info(plan)
    assert info.n_buckets == 5 and info.shard == 15_554_976 and info.phi_pad == 124_439_808
    Z.zero_plan_destroy(plan)
    w = W.workload(4)
    plan = _plan_for(w.sizes, w.n_d, w.stage, 0, w.unit_first)
    assert Z.zero_plan_info(plan).shard == 842_301_952
    Z.zero_plan_destroy(plan)


@pytest.mark.parametrize("args,code", [
    (([4, 4], 0, 1), Z.ZERO_EINVAL),
    (([4, 4], 4, 4), Z.ZERO_EINVAL),
    (([4, -1], 2, 1), Z.ZERO_EINVAL),
    (([4, 4], Z.ZERO_MAX_RANKS + 1, 1), Z.ZERO_ERANGE),
])
def test_plan_create_errors(args, code):
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_plan_create(*args)
    assert e.value.status == code


def test_plan_create_argument_errors():
    for kw, code in [(dict(stage=3, bucket_elems=8), Z.ZERO_EINVAL),
                     (dict(stage=1, unit_first=[0, 1]), Z.ZERO_EINVAL),
                     (dict(stage=3, unit_first=[1]), Z.ZERO_EINVAL),
                     (dict(stage=3, unit_first=[0, 2, 2]), Z.ZERO_EINVAL),
                     (dict(stage=2, dtype16=7), Z.ZERO_EINVAL),
                     (dict(stage=2, bucket_elems=-1), Z.ZERO_EINVAL)]:
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_plan_create([3, 5, 7], 2, **kw)
        assert e.value.status == code, kw
        assert Z.zero_last_error()


def test_calls_out_of_order_fail_without_touching_the_gpu():
    plan = _plan_for([10, 20], 3, 2, 8)
    try:
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_step_finish(plan)
        assert e.value.status == Z.ZERO_ESTATE
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_gather_layer(plan, 0, 0x1000)
        assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:     # nothing bound yet
            Z.zero_step(plan, [0x1000] * 3, 0, Z.hyper())
        assert e.value.status == Z.ZERO_ESTATE
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_step(plan, [0x1000] * 2, 0, Z.hyper())
        assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_bind_peer(plan, 0, 0x1000)
        assert e.value.status == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_plan_tables(plan, 99)
        assert e.value.status == Z.ZERO_EINVAL
        buf = (ctypes.c_int64 * 1)()
        n = ctypes.c_int64()
        assert Z.lib().zero_plan_tables(plan, Z.ZERO_TABLE_SHARD_SEGMENTS, buf, 1, ctypes.byref(n)) \
            == Z.ZERO_ERANGE
    finally:
        Z.zero_plan_destroy(plan)


def test_execution_options_are_checked_on_the_host():
    """zero_set_option / zero_get_option: defaults, values outside their ranges give EINVAL; a
    staging ring (stages x tile x (2 N_d + 12) bytes + 384 bytes) beyond one block's 227 KB of
    shared memory gives ERANGE and leaves the earlier geometry in place."""
    plan = _plan_for([10, 20], 7, 2, 8)
    try:
        assert Z.zero_get_option(plan, Z.ZERO_OPT_STAGING) == Z.ZERO_STAGING_AUTO
        assert Z.zero_get_option(plan, Z.ZERO_OPT_WAIT_LIMIT_NS) == 1_000_000_000
        assert Z.zero_get_option(plan, Z.ZERO_OPT_BULK_TILE) == 2048      # 2048 x 26 B <= 53.5 KB
        assert Z.zero_get_option(plan, Z.ZERO_OPT_BULK_STAGES) == 2
        assert Z.zero_get_option(plan, Z.ZERO_OPT_LAST_STEP_KERNEL) == -1
        assert Z.zero_get_option(plan, Z.ZERO_OPT_HOST_PIPELINE) == 1
        assert Z.zero_get_option(plan, Z.ZERO_OPT_OFFLOAD_DEFER) == 0
        assert Z.zero_get_option(plan, Z.ZERO_OPT_UNIT_ORDER) == 0
        assert Z.zero_get_option(plan, Z.ZERO_OPT_LAST_GATHER_IN_STEP) == -1
        assert Z.zero_get_option(plan, Z.ZERO_OPT_HOST_H2D_BYTES) == 0
        assert Z.zero_get_option(plan, Z.ZERO_OPT_HOST_D2H_BYTES) == 0
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_get_option(plan, 99)
        assert e.value.status == Z.ZERO_EINVAL
        for opt, val in ((Z.ZERO_OPT_STAGING, 3), (Z.ZERO_OPT_STAGING, -1),
                         (Z.ZERO_OPT_WAIT_LIMIT_NS, -1), (Z.ZERO_OPT_BULK_TILE, 12),
                         (Z.ZERO_OPT_BULK_TILE, 16384), (Z.ZERO_OPT_BULK_TILE, 4),
                         (Z.ZERO_OPT_BULK_STAGES, 1), (Z.ZERO_OPT_BULK_STAGES, 17), (99, 0),
                         (Z.ZERO_OPT_HOST_PIPELINE, 2), (Z.ZERO_OPT_HOST_H2D_BYTES, 0),
                         (Z.ZERO_OPT_HOST_D2H_BYTES, 0), (Z.ZERO_OPT_LAST_STEP_KERNEL, 0),
                         (Z.ZERO_OPT_LAST_GATHER_IN_STEP, 1), (Z.ZERO_OPT_OFFLOAD_DEFER, 2),
                         (Z.ZERO_OPT_UNIT_ORDER, 2), (Z.ZERO_OPT_UNIT_ORDER, -1)):
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_set_option(plan, opt, val)
            assert e.value.status == Z.ZERO_EINVAL, (opt, val)
        for opt, val in ((Z.ZERO_OPT_STAGING, 1), (Z.ZERO_OPT_STAGING, 2), (Z.ZERO_OPT_STAGING, 0),
                         (Z.ZERO_OPT_HOST_PIPELINE, 0), (Z.ZERO_OPT_HOST_PIPELINE, 1),
                         (Z.ZERO_OPT_OFFLOAD_DEFER, 1), (Z.ZERO_OPT_OFFLOAD_DEFER, 0),
                         (Z.ZERO_OPT_UNIT_ORDER, 1), (Z.ZERO_OPT_UNIT_ORDER, 0),
                         (Z.ZERO_OPT_WAIT_LIMIT_NS, 0), (Z.ZERO_OPT_BULK_TILE, 4096),
                         (Z.ZERO_OPT_BULK_TILE, 1024), (Z.ZERO_OPT_BULK_STAGES, 8)):
            Z.zero_set_option(plan, opt, val)
        # 1024 x 26 B = 26 KB per buffer: 8 fit, 16 do not
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_set_option(plan, Z.ZERO_OPT_BULK_STAGES, 16)
        assert e.value.status == Z.ZERO_ERANGE
        # 8192 x 26 B = 208 KB per buffer: two do not fit
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_set_option(plan, Z.ZERO_OPT_BULK_TILE, 8192)
        assert e.value.status == Z.ZERO_ERANGE
        Z.zero_set_option(plan, Z.ZERO_OPT_BULK_STAGES, 0)     # automatic: 2 buffers of 104 KB
        Z.zero_set_option(plan, Z.ZERO_OPT_BULK_TILE, 4096)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_set_option(plan, Z.ZERO_OPT_BULK_STAGES, 3)
        assert e.value.status == Z.ZERO_ERANGE
    finally:
        Z.zero_plan_destroy(plan)
    plan = _plan_for([10], 1, 1)
    try:                                     # N_d = 1: 8192 x 14 B x 2 + 256 B fit in 227 KB
        Z.zero_set_option(plan, Z.ZERO_OPT_BULK_TILE, 8192)
        Z.zero_set_option(plan, Z.ZERO_OPT_BULK_STAGES, 2)
    finally:
        Z.zero_plan_destroy(plan)


def test_gather_options_are_checked_on_the_host():
    """The gather's kernel, bulk-copy chunk (a multiple of 8 elements up to 32768) and ring
    entries (3 to 32); a ring of entries x chunk x 2 B + 384 B beyond 227 KB gives ERANGE
    and leaves the earlier geometry in place."""
    plan = _plan_for([10, 20], 4, 3, 0)
    try:
        assert Z.zero_get_option(plan, Z.ZERO_OPT_GATHER_STAGING) == Z.ZERO_STAGING_AUTO
        assert Z.zero_get_option(plan, Z.ZERO_OPT_GATHER_CHUNK) == 16384
        assert Z.zero_get_option(plan, Z.ZERO_OPT_GATHER_STAGES) == 4
        for opt, val in ((Z.ZERO_OPT_GATHER_STAGING, 3), (Z.ZERO_OPT_GATHER_STAGING, -1),
                         (Z.ZERO_OPT_GATHER_CHUNK, 4), (Z.ZERO_OPT_GATHER_CHUNK, 12),
                         (Z.ZERO_OPT_GATHER_CHUNK, 32776), (Z.ZERO_OPT_GATHER_STAGES, 2),
                         (Z.ZERO_OPT_GATHER_STAGES, 33), (Z.ZERO_OPT_GATHER_STAGES, -1)):
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_set_option(plan, opt, val)
            assert e.value.status == Z.ZERO_EINVAL, (opt, val)
        for val in (0, 1, 2):
            Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_STAGING, val)
            assert Z.zero_get_option(plan, Z.ZERO_OPT_GATHER_STAGING) == val
        Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_CHUNK, 8)
        Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_STAGES, 32)
        Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_STAGES, 0)
        Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_CHUNK, 8192)            # 4 x 16 KB
        with pytest.raises(Z.ZeroError) as e:                              # 4 x 64 KB
            Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_CHUNK, 32768)
        assert e.value.status == Z.ZERO_ERANGE
        assert Z.zero_get_option(plan, Z.ZERO_OPT_GATHER_CHUNK) == 8192
        Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_STAGES, 13)             # 13 x 16 KB = 208 KB
        with pytest.raises(Z.ZeroError) as e:                              # 15 x 16 KB = 240 KB
            Z.zero_set_option(plan, Z.ZERO_OPT_GATHER_STAGES, 15)
        assert e.value.status == Z.ZERO_ERANGE
        assert Z.zero_get_option(plan, Z.ZERO_OPT_GATHER_STAGES) == 13
    finally:
        Z.zero_plan_destroy(plan)


def test_empty_model_plan():
    plan = _plan_for([], 4, 2, 0)
    info = Z.zero_plan_info(plan)
    assert info.phi == info.phi_pad == info.shard == info.n_buckets == 0
    assert Z.zero_plan_tables(plan, Z.ZERO_TABLE_SHARD_SEGMENTS) == []
    Z.zero_plan_destroy(plan)


# ---------------------------------------------------------------------- FSDP-2 per-parameter plans

def _compare_per_param(sizes, dim0, n_d, units):
    plan = Z.zero_plan_create_per_param(sizes, dim0, n_d, units or None)
    try:
        pp = oracle.PerParam(sizes, dim0, n_d, units or None)
        rows = Z.zero_plan_tables(plan, Z.ZERO_TABLE_PARAM_CHUNKS)
        assert [r[:9] for r in rows] == [tuple(int(x) for x in c) for c in pp.chunks]
        info = Z.zero_plan_info(plan)
        assert info.shard == pp.per_rank and info.phi == info.phi_pad == sum(sizes)
        ut = Z.zero_plan_tables(plan, Z.ZERO_TABLE_UNITS)
        assert [u[2] for u in ut] == pp.unit_numel and [u[5] for u in ut] == list(pp.unit_base[:-1])
        for r in range(n_d):
            elems = Z.zero_rank_state_elems(plan, r)
            end = 0
            for row in rows:
                if row[0] != r:
                    continue
                phys, local = row[9], row[6] * row[5]
                assert phys >= end and phys - end < 8 and (phys - row[7]) % 8 == 0
                end = phys + local
            assert end <= elems and elems % 8 == 0
        with pytest.raises(Z.ZeroError):
            Z.zero_plan_tables(plan, Z.ZERO_TABLE_SHARD_SEGMENTS)
    finally:
        Z.zero_plan_destroy(plan)


def test_per_param_tables_match_oracle_random():
    rng = np.random.default_rng(50)
    for _ in range(200):
        nt = int(rng.integers(1, 10))
        dim0 = [int(x) for x in rng.integers(0, 30, size=nt)]
        sizes = [d * int(c) for d, c in zip(dim0, rng.integers(1, 9, size=nt))]
        units = []
        if nt > 1 and rng.random() < 0.6:
            units = [0] + sorted(set(int(x) for x in rng.integers(1, nt, size=2)))
        _compare_per_param(sizes, dim0, int(rng.integers(1, 17)), units)


@pytest.mark.parametrize("i", [2, 3, 4])
def test_per_param_tables_match_oracle_workloads(i):
    w = W.per_param_variant(W.workload(i))
    _compare_per_param(list(w.sizes), list(w.dim0), w.n_d, list(w.unit_first))


def test_per_param_argument_errors():
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_plan_create_per_param([10, 7], [3, 7], 2)         # 10 is not a multiple of 3
    assert e.value.status == Z.ZERO_EINVAL
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_plan_create_per_param([0, 7], [0, 7], 0)
    assert e.value.status == Z.ZERO_EINVAL


_EXHAUSTION_CHILD = """
import ctypes, resource, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import zero_sharded_mixed_03_gb300 as Z
L = Z.lib()
n = 20_000_000
sizes = np.ones(n, dtype=np.int64)
out = ctypes.c_void_p()
vm = int(open('/proc/self/statm').read().split()[0]) * resource.getpagesize()
soft, hard = resource.getrlimit(resource.RLIMIT_AS)
resource.setrlimit(resource.RLIMIT_AS, (vm + (256 << 20), hard))
st = L.zero_plan_create(sizes.ctypes.data, n, 8, 2, 0, None, 0, 0, ctypes.byref(out))
resource.setrlimit(resource.RLIMIT_AS, (soft, hard))
print(st, out.value is None, L.zero_last_error().decode())
"""


def test_host_exhaustion_is_reported_not_thrown():
    """A plan whose host tables do not fit (20M tensors under an address-space limit just above
    the process's current use, in a child process): zero_plan_create returns ZERO_ENOMEM with a
    message and no plan, instead of letting std::bad_alloc cross the C ABI (which would abort
    the process)."""
    import subprocess
    import sys
    if not os.path.exists("/proc/self/statm"):
        pytest.skip("needs /proc")
    run = subprocess.run([sys.executable, "-c", _EXHAUSTION_CHILD, ROOT], capture_output=True,
                         text=True, timeout=300)
    assert run.returncode == 0, run.stderr[-2000:]
    status, no_plan, msg = run.stdout.strip().split(" ", 2)
    assert int(status) == Z.ZERO_ENOMEM and no_plan == "True", run.stdout
    assert "host resource exhausted" in msg



def test_unit_slice_keeps_one_unit_of_a_stage3_workload():
    """The profiling slice of a stage-3 workload: the tensors (and dim-0 sizes) of one unit, as
    a one-unit workload; the library's plan of the slice has that unit's padded size."""
    w = W.workload(3)
    first, count = w.units()[1]
    s = W.unit_slice(w, 1)
    assert s.sizes == w.sizes[first:first + count] and s.unit_first == (0,) and s.inject is None
    assert s.phi == 50_358_272                         # one 2048-wide GPT block
    plan = _plan_for(s.sizes, s.n_d, 3, 0, [0])
    try:
        info = Z.zero_plan_info(plan)
        assert info.n_units == 1 and info.phi_pad == s.phi   # divisible by N_d = 16: no padding
    finally:
        Z.zero_plan_destroy(plan)
    pp = W.unit_slice(W.per_param_variant(W.workload(4)), 1)
    f4, c4 = W.workload(4).units()[1]
    assert pp.dim0 == W.per_param_variant(W.workload(4)).dim0[f4:f4 + c4] and pp.per_param
    with pytest.raises(ValueError):
        W.unit_slice(W.workload(1), 0)                 # stage 2: no units


def test_host_staging_size_and_host_path_state_errors():
    """info.host_staging_bytes = N_d areas of the largest call's range rounded up to a multiple
    of 8 elements, 2 bytes each; the host-buffer calls refuse an unbound plan (no GPU needed)."""
    for sizes, n_d, stage, bucket, units in (([10, 20, 7], 3, 2, 9, None), ([1000], 4, 1, 0, None),
                                             ([5, 6, 7, 8], 2, 3, 0, [0, 2])):
        plan = _plan_for(sizes, n_d, stage, bucket, units)
        try:
            info = Z.zero_plan_info(plan)
            assert info.host_staging_bytes == n_d * (-(-info.max_contrib_elems // 8) * 8) * 2
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_bind_host_staging(plan, [16, 4096], info.host_staging_bytes)
            assert e.value.status == Z.ZERO_ESTATE               # no rank bound yet
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_step_host(plan, [16] * n_d, 0, Z.hyper(), 16)
            assert e.value.status == Z.ZERO_ESTATE
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_step_host_finish(plan)
            assert e.value.status == Z.ZERO_ESTATE               # no host call in the step
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_step_host(plan, [16] * (n_d + 1), 0, Z.hyper(), 16)
            assert e.value.status == Z.ZERO_EINVAL
        finally:
            Z.zero_plan_destroy(plan)
