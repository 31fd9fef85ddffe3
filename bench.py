#!/usr/bin/env python3
"""Throughput of the sharded mixed-precision AdamW step on GB300.

One step = one pass of the whole hot path over one step's synthetic gradients: for every
reduce-scatter bucket (stages 1/2) or FSDP unit (stage 3: all-gather of the unit first) the
fused reduce + unscale + inf/nan flag + AdamW + 16-bit cast kernel, then the commit/skip
decision.  Default workload: ZeRO-3 per layer over a 1.3B-parameter GPT (24 blocks, d = 2048, ffn 8192,
vocab 50257; 26 units), N_d = 16 emulated ranks.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the same workload.
"""
from __future__ import annotations

import argparse
import importlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ZeRO step params updated/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "params/s"
DEFAULT_CONFIG = 3
DEFAULT_STAGING = "auto"
FALLBACK_HBM_GBS = 6800.0
# GB300's rated HBM3e bandwidth per GPU (nominal, ~7.9 TB/s), reported beside the measured
# copy bandwidth that the roofline fractions use as their peak
NOMINAL_HBM_GBS = 7900.0
# Gradient sets rotated through the timed steps.  A backward pass rewrites the same gradient
# buffers every step, so a few persistent sets model training; each step still reads inputs
# it did not read the step before, and every set is far larger than the 129 MB L2.  (Cycling
# through tens of GB of distinct sets instead measures GPU TLB reach, not the step.)
ROTATE_SETS = 4

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the step kernel from
# one ncu capture, per (workload, kernel), valid only for the kernel source it was taken on
# (first 16 hex digits of the SHA-256 of zero_kernels.cuh, the device code); reported as null
# once that source changes.
MEASURED_TRAFFIC = {(1, "bulk_step_kernel"): ("1087b358f163289b", 2_286_208_768),
                    # one launch captured (bucket 0 of 5), scaled by elements to the average
                    # launch the bench times
                    (2, "bulk_step_kernel"): ("1087b358f163289b", 1_003_294_020),
                    # the step launch that also gathers the next unit (one launch captured on
                    # a two-unit slice of the model, scaled by algorithmic bytes to the average
                    # launch of the full step)
                    (3, "bulk_step_kernel + gather"): ("1087b358f163289b", 3_068_613_361),
                    (4, "bulk_step_kernel + gather"): ("1087b358f163289b", 1_765_648_613)}
KERNEL_SOURCE = os.path.join(ROOT, "zero_sharded_mixed_03_gb300", "csrc", "zero_kernels.cuh")


def kernel_source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the kernel source (the traffic records' key)."""
    import hashlib
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(config: int, kernel: str):
    import hashlib
    rec = MEASURED_TRAFFIC.get((config, kernel))
    if rec is None:
        return None
    with open(KERNEL_SOURCE, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    return rec[1] if digest == rec[0] else None


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-elems", type=int, default=4_194_304)
    ap.add_argument("--mem-budget-gb", type=float, default=160.0)
    ap.add_argument("--no-graph", action="store_true",
                    help="enqueue the timed steps one by one instead of replaying them as one "
                         "captured CUDA graph")
    ap.add_argument("--offload", action="store_true",
                    help="ZeRO-Offload: gradients reduced on the GPU into pinned host memory, AdamW "
                         "on the host CPU threads, 16-bit parameters copied back")
    ap.add_argument("--offload-defer", action="store_true",
                    help="with --offload: ZERO_OPT_OFFLOAD_DEFER (the contribution buffers stay "
                         "unchanged until the finish, so every bucket's flag pass runs first and "
                         "the reductions stream to the host while it updates)")
    ap.add_argument("--per-param", action="store_true",
                    help="FSDP-2 per-parameter (dim-0) sharding of the same model")
    ap.add_argument("--overlap", action="store_true",
                    help="stage 3: gather unit u+1 on a second stream while unit u steps "
                         "(zero_step_units_overlapped); no per-launch events in this mode")
    ap.add_argument("--schedule", choices=["fused", "serial"], default="fused",
                    help="stage 3: fused (default): unit u's step launch also gathers unit u+1 "
                         "(zero_step_gather_next; unit 0 is gathered on its own); serial: every "
                         "unit's gather as a launch of its own before its step")
    ap.add_argument("--unit-order", choices=["asc", "desc"], default="asc",
                    help="stage 3: step the units first to last (default), or last to first as "
                         "a backward pass produces their gradients (ZERO_OPT_UNIT_ORDER)")
    ap.add_argument("--staging", choices=["auto", "ldg", "bulk"], default=DEFAULT_STAGING,
                    help="bulk: cp.async.bulk (TMA) staging of the contribution and state tiles "
                         "into shared memory; ldg: 128-bit register loads; auto (default): the "
                         "library's choice (staged where its residency pays off)")
    ap.add_argument("--n-d", type=int, default=0,
                    help="override the workload's N_d (kernel sweeps; 0: the workload's own)")
    ap.add_argument("--bulk-tile", type=int, default=0, help="bulk staging: elements per tile")
    ap.add_argument("--bulk-stages", type=int, default=0, help="bulk staging: ring depth")
    ap.add_argument("--gather-staging", choices=["default", "ldg", "bulk"], default="default",
                    help="stage-3 gather kernel: register loads or bulk-staged (default: the plan's)")
    ap.add_argument("--gather-chunk", type=int, default=0, help="bulk gather: elements per copy")
    ap.add_argument("--gather-stages", type=int, default=0, help="bulk gather: ring entries")
    ap.add_argument("--profile-unit", type=int, default=None,
                    help="stage 3: restrict the workload to this one unit (for ncu captures of a "
                         "few GB; not the benchmark workload)")
    ap.add_argument("--profile-units", type=int, default=1,
                    help="with --profile-unit: this many units from it (2: one step launch that "
                         "also gathers the next unit)")
    ap.add_argument("--grad-norm", choices=["off", "report", "clip"], default="off",
                    help="report: global gradient norm inside the fused pass; clip: norm pre-pass "
                         "over every bucket/unit, then the update clipped at max norm 1.0")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, dist=None) -> float:
    """Largest value over the ranks of the (optional) process group: the job's wall time is
    the slowest replica's.  NCCL reduces a CUDA tensor, gloo a CPU one."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(elems_per_step: int, applied_steps: int, world: int, seconds: float) -> float:
    """Whole-job throughput of N independent replicas: every rank updates elems_per_step
    parameters per applied step; the job takes the slowest rank's time."""
    return world * elems_per_step * applied_steps / seconds


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML every ~0.5 ms while the timed region
    runs (a short run's timed region lasts milliseconds, under nvidia-smi's sampling period).
    Reads only; the device is found by its UUID, so CUDA_VISIBLE_DEVICES does not matter."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, cuda_index: int):
        import ctypes
        import threading
        self.ctypes, self.threading = ctypes, threading
        self.ok, self.samples, self.thread, self.running = False, [], None, False
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            uuid = str(getattr(torch.cuda.get_device_properties(cuda_index), "uuid", "") or "")
            if uuid:
                key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                rc = nv.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(self.handle))
            else:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.handle))
            if rc != 0:
                return
            self.reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.ok = nv, True
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0 else None
        except Exception:
            self.ok = False

    def _run(self):
        ctypes = self.ctypes
        mhz, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        while self.running:
            if (self.nv.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0 and
                    self.reasons(self.handle, ctypes.byref(bits)) == 0):
                self.samples.append((float(mhz.value), int(bits.value)))
            time.sleep(0.0005)

    def start(self):
        if self.ok:
            self.running = True
            self.thread = self.threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def stop(self):
        if not self.ok or self.thread is None:
            return None
        self.running = False
        self.thread.join()
        if not self.samples:
            return None
        reasons = sorted({name for _, b in self.samples for bit, name in self.REASONS.items() if b & bit})
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml, timed region"}


# ----------------------------------------------------------------------------- GPU arm

class Bench:
    """A workload bound to the product API with pre-generated contribution sets."""

    def __init__(self, w, mem_budget_gb: float, n_sets_wanted: int, grad_norm: str = "off",
                 options=None, fused_gather: bool = False, unit_order: str = "asc"):
        import torch
        import synth
        import zero_sharded_mixed_03_gb300 as Z
        from synth.fill import fill_device
        from synth.run import Run

        self.torch, self.Z, self.synth = torch, Z, synth
        self.w = w
        self.fused_gather = fused_gather and w.stage == 3 and not w.offload
        self.gather_in_step = None            # learnt from the library on the first step
        # plan, state, 16-bit buffers, initial params
        self.run = Run(w, alloc_contribs=False, options=options)
        self.g = self.run.g
        self.units = self.run.units
        self.info = self.run.info
        self.bound = self.run.bound
        self.all_bound = len(self.bound) == w.n_d
        self.calls = self.run.ranges()
        if unit_order == "desc" and w.stage == 3:
            # last unit first: the order of every per-call loop below, the compact contribution
            # layout included; the whole-step call takes the same order as an option
            self.calls = self.calls[::-1]
            self.g.set_option(Z.ZERO_OPT_UNIT_ORDER, 1)
        # Contribution layout of one step: for each call the slices the bound ranks read.
        # All ranks bound: the call's whole range.  Otherwise: each bound rank's shard slice.
        self.read_spans = []          # per call: list of (flat lo, flat hi, compact offset)
        off = 0
        for which, lo, hi in self.calls:
            spans = []
            if self.all_bound:
                spans.append((lo, hi, off, 0))
                off += hi - lo
            elif w.per_param:
                # a rank's rows are spread over the whole unit: every unit reuses one
                # unit-sized buffer per contributing rank
                spans.append((lo, hi, 0, 0))
                off = max(off, hi - lo)
            else:
                for r in sorted(self.bound):
                    if w.stage == 3:
                        U = self.units[which]
                        a, e = U[5] + r * U[4], U[5] + (r + 1) * U[4]
                    else:
                        S = self.units[0][4]
                        a, e = max(lo, r * S), min(hi, (r + 1) * S)
                    if a < e:
                        spans.append((a, e, off, a - lo))
                        off += e - a
                # one base pointer per contribution: a compact layout serves one bound rank
                assert len(spans) <= 1, "compact contributions need a single bound rank"
            self.read_spans.append(spans)
        self.set_elems = off
        set_bytes = off * 2 * w.n_d
        self.n_sets = int(max(1, min(n_sets_wanted, (mem_budget_gb * 1e9) // max(1, set_bytes))))
        self.sets = []
        for s in range(self.n_sets):
            bufs = [torch.empty(max(8, off), dtype=torch.int16, device="cuda") for _ in range(w.n_d)]
            for r in range(w.n_d):
                st = synth.grad_stream(w, s + 1, r, planted=False)   # no skip in the rotation
                for spans in self.read_spans:
                    for (a, e, o, _rel) in spans:
                        fill_device(bufs[r][o:o + (e - a)], st, self.units, a, e)
            self.sets.append(bufs)
        torch.cuda.synchronize()
        self.elems_per_step = int(self.info.shard) * len(self.bound)
        self.bytes_per_elem = 2 * w.n_d + 26
        self.hyper = self.run.hyper
        self._count_launches()
        self.clip = grad_norm == "clip"
        if grad_norm != "off":
            h = self.hyper
            self.hyper = Z.hyper(h.lr, h.beta1, h.beta2, h.eps, h.weight_decay,
                                 1.0 if self.clip else 0.0, grad_norm == "report")

    def _count_launches(self):
        """Kernel launches per step, from the plan's work items: one launch per 32 items (256
        when a call has more than 32), per call; gathers likewise per copied shard or chunk."""
        def launches(items):
            return 0 if items == 0 else (1 if items <= 32 else -(-items // 256))
        bound = set(self.bound)
        w = self.w
        fused, gathers = [], []
        all_items = 0
        for which, lo, hi in self.calls:
            # element counts of the call's work items, in the library's launch order
            if w.per_param:
                sizes = [c[4] * c[5] for c in self.g.chunks if c[1] == which and c[4] > 0 and c[0] in bound]
                copies = sum(1 for c in self.g.chunks if c[1] == which and c[4] > 0)
            elif w.stage == 3:
                shard = self.units[which][4]
                sizes = [shard for r in sorted(bound)] if shard > 0 else []
                copies = w.n_d if shard > 0 else 0
            else:
                S = self.units[0][4]
                sizes = [min(hi, (r + 1) * S) - max(lo, r * S) for r in sorted(bound)
                         if max(lo, r * S) < min(hi, (r + 1) * S)]
                copies = 0
            items = len(sizes)
            all_items += items if w.stage == 3 else 0
            if w.offload:
                # a flag-only pass over the call, then the writing reduction in groups of
                # items of >= 4M elements, each group launched in pieces of the call's capacity
                cap = 32 if items <= 32 else 256
                n = launches(items)
                k = 0
                while k < items:
                    e, acc = k, 0
                    while e < items and acc < (1 << 22):
                        acc += sizes[e]
                        e += 1
                    n += -(-(e - k) // cap)
                    k = e
                fused.append(n)
            else:
                fused.append(launches(items))
            gathers.append(launches(copies))
        if w.stage != 3:
            all_items = len(bound)
        self.fused_launches, self.gather_launches = fused, gathers
        # offloaded plans re-cast on the host: no re-cast kernel
        self.recast_launches = 0 if w.offload else launches(all_items)

    def call_ptrs(self, bufs, ci):
        """Per-rank contribution pointers of call ci: base such that base + c_off hits the slice."""
        spans = self.read_spans[ci]
        if not spans:
            return [bufs[r].data_ptr() for r in range(self.w.n_d)]
        a, e, o, rel = spans[0]
        # compact slice o holds flat [a, e), which the kernel addresses as call offset `rel`
        return [bufs[r].data_ptr() + 2 * (o - rel) for r in range(self.w.n_d)]

    def step_overlapped(self, bufs, comm, wait=False):
        """Whole stage-3 step through zero_step_units_overlapped; returns (result, launches)."""
        gb = self.gather_bufs()
        # unit-major pointers (unit u's contributions at [u * N_d]), whatever the call order
        by_unit = sorted(range(len(self.calls)), key=lambda ci: self.calls[ci][0])
        ptrs = [p for ci in by_unit for p in self.call_ptrs(bufs, ci)]
        res = self.Z.zero_step_units_overlapped(
            self.g.plan, ptrs, [b.data_ptr() for b in gb], self.hyper,
            self.torch.cuda.current_stream().cuda_stream, comm.cuda_stream, wait)
        launches = ((1 + self.clip) * sum(self.fused_launches) + sum(self.gather_launches)
                    + self.recast_launches + (0 if self.recast_launches else 1))
        return res, launches

    def gather_bufs(self):
        if not hasattr(self, "_gbufs"):
            n = max(8, int(self.info.max_unit_pad))
            self._gbufs = [self.torch.empty(n, dtype=self.torch.int16, device="cuda") for _ in range(2)]
        return self._gbufs

    def step_fused(self, bufs, events=None, gather_events=None, wait=False):
        """One stage-3 step in which unit u's step launch also gathers unit u+1
        (zero_step_gather_next); unit 0 is gathered by a launch of its own.  Events as in step();
        the gather pairs then time only unit 0's gather.  Returns (result, launches)."""
        gb = self.gather_bufs()
        launches = 0
        n = len(self.calls)
        if self.clip:                    # the norm over every unit before any step
            for ci, (which, lo, hi) in enumerate(self.calls):
                self.g.grad_norm(self.call_ptrs(bufs, ci), which)
                launches += self.fused_launches[ci]
        if gather_events is not None:
            a, c = next(gather_events)
            a.record()
        self.g.gather(self.calls[0][0], gb[0])
        if gather_events is not None:
            c.record()
        launches += self.gather_launches[0]
        for ci, (which, lo, hi) in enumerate(self.calls):
            self.g.release(which)
            if events is not None:
                a, c = next(events)
                a.record()
            if ci + 1 < n:
                self.g.step_gather_next(self.call_ptrs(bufs, ci), which, self.hyper,
                                        self.calls[ci + 1][0], gb[(ci + 1) % 2])
                if self.gather_in_step is None:
                    self.gather_in_step = self.Z.zero_get_option(
                        self.g.plan, self.Z.ZERO_OPT_LAST_GATHER_IN_STEP) == 1
                if not self.gather_in_step:
                    launches += self.gather_launches[ci + 1]
            else:
                self.g.step(self.call_ptrs(bufs, ci), which, self.hyper)
            if events is not None:
                c.record()
            launches += self.fused_launches[ci]
        res = self.g.finish(wait=wait)
        launches += self.recast_launches + (0 if self.recast_launches else 1)
        return res, launches

    def step(self, bufs, events=None, gather_events=None, wait=False):
        """Enqueue one step; with wait=True also read the step result back (synchronises).

        events / gather_events: iterators of pre-created (start, end) CUDA event pairs recorded
        around each fused launch / gather launch.  Returns (result or None, kernel launches).
        """
        if self.fused_gather:
            return self.step_fused(bufs, events, gather_events, wait)
        launches = 0
        if self.clip:
            for ci, (which, lo, hi) in enumerate(self.calls):
                self.g.grad_norm(self.call_ptrs(bufs, ci), which)
                launches += self.fused_launches[ci]
        for ci, (which, lo, hi) in enumerate(self.calls):
            if self.w.stage == 3:
                if gather_events is not None:
                    a, c = next(gather_events)
                    a.record()
                self.g.gather(which, self.run.gather_buf)
                if gather_events is not None:
                    c.record()
                self.g.release(which)
                launches += self.gather_launches[ci]
            if events is not None:
                a, c = next(events)
                a.record()
            self.g.step(self.call_ptrs(bufs, ci), which, self.hyper)
            if events is not None:
                c.record()
            launches += self.fused_launches[ci]
        res = self.g.finish(wait=wait)
        # the re-cast kernel(s) (which return at once unless the step was skipped); the last one
        # also commits (a separate commit launch only when there is nothing to re-cast)
        launches += self.recast_launches + (0 if self.recast_launches else 1)
        return res, launches


def measure(b, args, torch, overlap, comm, use_graph, dist, pairs, sample_clocks=False,
            launch_events=True):
    """Time args.steps steps between barrier/synchronise brackets: captured once as a CUDA
    graph and replayed, or enqueued one by one.  launch_events: timing events captured as graph
    nodes around every step / gather launch (instrumentation for the per-launch roofline; the
    whole-step figures come from a region without them).  Returns the region's ms, the
    per-launch ms of the step and gather kernels, the launch count and (sample_clocks) the
    NVML clock samples."""
    w = b.w
    n_calls = args.steps * len(b.calls)
    fused_pairs = pairs(n_calls, use_graph) if (not overlap and launch_events) else []
    n_gathers = args.steps if b.fused_gather else n_calls
    gather_pairs = (pairs(n_gathers, use_graph)
                    if (w.stage == 3 and not overlap and launch_events) else [])
    ev_fused, ev_gather = iter(fused_pairs), iter(gather_pairs)
    launches = 0

    def timed_steps():
        nonlocal launches
        for k in range(args.steps):
            bufs = b.sets[(args.warmup + k) % b.n_sets]
            if overlap:
                _, n = b.step_overlapped(bufs, comm)
            elif launch_events:
                _, n = b.step(bufs, ev_fused, ev_gather if w.stage == 3 else None)
            else:
                _, n = b.step(bufs)
            launches += n

    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                timed_steps()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    region = NvmlSampler(torch.cuda.current_device()) if sample_clocks else None
    if region:
        region.start()
    t0.record()
    if graph is not None:
        graph.replay()
    else:
        timed_steps()
    t1.record()
    torch.cuda.synchronize()
    region_clk = region.stop() if region else None
    ms = t0.elapsed_time(t1)
    if dist:
        ms = max_over_ranks(ms, dist)
    return {"ms": ms, "fused_ms": [x.elapsed_time(y) for x, y in fused_pairs],
            "gather_ms": [x.elapsed_time(y) for x, y in gather_pairs], "launches": launches,
            "region_clk": region_clk, "graph": graph is not None}


def gpu_arm(args, world, rank, local):
    import torch
    from synth import workloads as W
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = W.workload(args.config)
    if args.n_d:
        import dataclasses
        w = dataclasses.replace(w, n_d=args.n_d, name=f"{w.name} at N_d = {args.n_d}",
                                bound_ranks=None, inject=None)
    if args.per_param:
        w = W.per_param_variant(w)
    if args.profile_unit is not None:
        w = W.unit_slice(w, args.profile_unit, args.profile_units)
    if args.offload:
        import dataclasses
        w = dataclasses.replace(w, offload=True)
    Z = importlib.import_module("zero_sharded_mixed_03_gb300")
    staging = {"ldg": Z.ZERO_STAGING_REGISTER_LOADS, "bulk": Z.ZERO_STAGING_BULK,
               "auto": Z.ZERO_STAGING_AUTO}[args.staging]
    options = {Z.ZERO_OPT_STAGING: staging, Z.ZERO_OPT_BULK_TILE: args.bulk_tile,
               Z.ZERO_OPT_BULK_STAGES: args.bulk_stages}
    if args.offload and args.offload_defer:
        options[Z.ZERO_OPT_OFFLOAD_DEFER] = 1
    # gather ring: entries first when the chunk grows, so that no intermediate ring overflows
    gather = [(Z.ZERO_OPT_GATHER_CHUNK, args.gather_chunk), (Z.ZERO_OPT_GATHER_STAGES, args.gather_stages)]
    options.update(dict(gather[::-1] if args.gather_chunk > 16384 else gather))
    if args.gather_staging != "default":
        options[Z.ZERO_OPT_GATHER_STAGING] = {"ldg": Z.ZERO_STAGING_REGISTER_LOADS,
                                             "bulk": Z.ZERO_STAGING_BULK}[args.gather_staging]
    b = Bench(w, args.mem_budget_gb, min(ROTATE_SETS, args.warmup + args.steps), args.grad_norm,
              options, fused_gather=args.schedule == "fused" and not args.overlap,
              unit_order=args.unit_order)
    peak, peak_kind = peaks()

    for k in range(args.warmup):
        b.step(b.sets[k % b.n_sets])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    schedule_note = None
    if b.fused_gather and b.gather_in_step is False:
        # the library ran the gathers as launches of their own (e.g. register-load step
        # kernel): time them as such, every gather between its own events
        b.fused_gather = False
        schedule_note = "serial: the library launched the gathers separately"

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    def pairs(n, external=False):
        kw = {"external": True} if external else {}
        return [(torch.cuda.Event(enable_timing=True, **kw), torch.cuda.Event(enable_timing=True, **kw))
                for _ in range(n)]
    overlap = args.overlap and w.stage == 3
    comm = torch.cuda.Stream() if overlap else None
    # Timed region: the K steps captured as one CUDA graph (the host does all enqueueing at
    # capture time), with timing events captured as graph nodes around every fused / gather
    # launch; --no-graph (or a torch without graph timing events) enqueues them step by step.
    # (offloaded steps synchronise with the host; a graph needs the bias table built by warm-up)
    use_graph = not args.no_graph and not w.offload and args.warmup > 0
    if use_graph:
        try:
            torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            use_graph = False
    skipped_before = b.g.step_state().skipped_total
    # the timed steps as a user runs them (no instrumentation between launches)
    m = measure(b, args, torch, overlap, comm, use_graph, dist, pairs, sample_clocks=True,
                launch_events=False)
    region_clk = m["region_clk"]
    if dist:
        dist.barrier()
    clk = clocks.stop()
    if region_clk is not None:               # samples taken inside the timed region
        if clk is not None:
            region_clk["nvidia_smi"] = clk
        clk = region_clk
    ms, launches = m["ms"], m["launches"]
    skipped = b.g.step_state().skipped_total - skipped_before
    # the same steps again with events around every launch: the per-launch kernel times
    mi = measure(b, args, torch, overlap, comm, use_graph, dist, pairs) if not overlap else m
    fused_ms, gather_ms = mi["fused_ms"], mi["gather_ms"]
    overlap_report = None
    if overlap:
        # the same steps with every unit's gather followed by its step on one stream: what the
        # second stream hides is the difference
        # (timed without per-launch events, like the overlapped steps; the gathers' own time
        # from the same serial steps with events around each launch)
        fg, b.fused_gather = b.fused_gather, False
        ser = measure(b, args, torch, False, None, use_graph, dist, pairs, launch_events=False)
        ser_i = measure(b, args, torch, False, None, use_graph, dist, pairs)
        b.fused_gather = fg
        g_ms = sum(ser_i["gather_ms"]) / args.steps
        hidden = ser["ms"] / args.steps - ms / args.steps
        frac = max(0.0, min(1.0, hidden / g_ms)) if g_ms > 0 else 0.0
        overlap_report = {"overlapped_ms_per_step": round(ms / args.steps, 3),
                          "serial_ms_per_step": round(ser["ms"] / args.steps, 3),
                          "serial_gather_ms_per_step": round(g_ms, 3),
                          "hidden_ms_per_step": round(hidden, 3),
                          "gather_hidden_fraction": round(frac, 4),
                          "gather_bytes_per_step": 4 * int(b.info.phi_pad),
                          "gather_bytes_hidden_per_step": int(frac * 4 * int(b.info.phi_pad))}

    applied = args.steps - skipped
    elems = b.elems_per_step
    value = job_value(elems, applied, world, ms / 1e3)
    step_bytes = elems * b.bytes_per_elem
    if args.grad_norm == "clip":                    # the norm pre-pass reads the gradients again
        step_bytes += elems * 2 * w.n_d
    gather_bytes = 4 * int(b.info.phi_pad) if w.stage == 3 else 0
    hbm_gbs = (step_bytes + gather_bytes) * args.steps / (ms / 1e3) / 1e9
    # dominant kernel: the fused step; algorithmic bytes per launch = elements x (2 N_d + 26)
    # (+ 4 bytes per element of the unit a launch also gathers, in the fused schedule)
    per_launch_elems = elems / max(1, len(b.calls))
    launch_bytes = per_launch_elems * b.bytes_per_elem
    fused_sched = b.fused_gather and not overlap
    in_step_gather_bytes = 0
    if fused_sched and b.gather_in_step:
        in_step_gather_bytes = 4 * sum(b.units[c[0]][3] for c in b.calls[1:])
        launch_bytes = (elems * b.bytes_per_elem + in_step_gather_bytes) / max(1, len(b.calls))
    avg_fused_s = statistics.mean(fused_ms) / 1e3 if fused_ms else float("nan")
    achieved = launch_bytes / avg_fused_s / 1e9
    # the step kernel the library launched (the staging option, the residency rule of the
    # automatic choice, norm-report steps)
    last = Z.zero_get_option(b.g.plan, Z.ZERO_OPT_LAST_STEP_KERNEL)
    kernel = "bulk_step_kernel" if last == 1 else "fused_step_kernel"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": measured_traffic(args.config, kernel + (" + gather" if fused_sched and b.gather_in_step else "")),
                "kernel_source_sha256": kernel_source_hash(),
                "peak_source": peak_kind, "kernel": kernel,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "nominal_peak": NOMINAL_HBM_GBS,
                "launch_bytes": int(launch_bytes), "avg_launch_us": round(avg_fused_s * 1e6, 2),
                "launches_timed": len(fused_ms)}
    if not fused_ms or w.offload:                   # overlapped / offloaded: no fused kernel
        roofline = None
    if w.offload:
        # host memory bounds an offloaded step: per parameter the GPU writes the fp32 gradient
        # (4 B), the host update reads master, m, v and the gradient (16 B) and writes master,
        # m, v and the 16-bit parameter (14 B), and the copy engines read that parameter back
        # (2 B): 36 B, against the host's own copy bandwidth measured here with the update's
        # threads
        host_peak = host_copy_gbs(b.g.offload_threads)
        achieved_host = elems * 36 * applied / (ms / 1e3) / 1e9
        roofline = {"bound": "host memory", "achieved": round(achieved_host, 1),
                    "peak": round(host_peak, 1), "unit": "GB/s",
                    "frac": round(achieved_host / host_peak, 4), "traffic": None,
                    "peak_source": f"measured here: torch CPU copy on {b.g.offload_threads} threads",
                    "kernel": "host AdamW (zero_offload_finish)"}
    if gather_ms and roofline is not None:
        gstaging = Z.zero_get_option(b.g.plan, Z.ZERO_OPT_GATHER_STAGING)
        standalone = ("gather_kernel" if gstaging == Z.ZERO_STAGING_REGISTER_LOADS
                      else "bulk_gather_kernel")
        if fused_sched and b.gather_in_step:
            # the gathers of units 1.. stream inside the step launches: their bytes move at the
            # launch's combined rate; unit 0's gather is a launch of its own
            roofline["kernel"] = "bulk_step_kernel + next unit's gather (zero_step_gather_next)"
            roofline["gather_in_step_launch"] = True
            roofline["gather_achieved_gbs"] = roofline["achieved"]
            roofline["in_step_gather_bytes_per_step"] = in_step_gather_bytes
            g0 = 4 * b.units[b.calls[0][0]][3]
            roofline["unit0_gather_gbs"] = round(g0 / (statistics.mean(gather_ms) / 1e3) / 1e9, 1)
            roofline["unit0_gather_kernel"] = standalone
        else:
            g_bytes = 4 * int(b.info.phi_pad) / len(b.calls)
            roofline["gather_achieved_gbs"] = round(g_bytes / (statistics.mean(gather_ms) / 1e3) / 1e9, 1)
            roofline["gather_kernel"] = standalone

    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms / args.steps,
           "ms_per_step_with_launch_events": mi["ms"] / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype":
           "fp16" if w.dtype == W.FP16 else "bf16", "data": "synthetic",
           "config": {"workload": w.name, "workload_index": args.config, "n_d": w.n_d,
                      "stage": w.stage, "phi": w.phi, "bucket_elems": w.bucket_elems,
                      "units": len(b.units), "bound_ranks": len(b.bound),
                      "elems_updated_per_step": elems, "bytes_per_param": b.bytes_per_elem,
                      "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB per step)",
                      "contribution_sets": b.n_sets, "grad_norm": args.grad_norm,
                      "overlap": overlap, "graph": m["graph"], "per_param": w.per_param,
                      "schedule": (("overlap" if overlap else (schedule_note or args.schedule))
                                   if w.stage == 3 else None),
                      "unit_order": args.unit_order if w.stage == 3 else None,
                      "offload": w.offload, "staging": args.staging,
                      "profile_unit": args.profile_unit,
                      "profile_units": args.profile_units if args.profile_unit is not None else None,
                      "offload_threads": b.g.offload_threads if w.offload else None,
                      "offload_defer": bool(w.offload and args.offload_defer)},
           "hbm_gbs": round(hbm_gbs, 1), "hbm_frac": round(hbm_gbs / peak, 4),
           "hbm_frac_of_nominal": round(hbm_gbs / NOMINAL_HBM_GBS, 4),
           "skipped_steps": skipped, "roofline": roofline, "gpu_launches": launches,
           "clocks": clk}
    if overlap_report is not None:
        out["overlap"] = overlap_report

    # the end-to-end and CPU legs report a failure in the line instead of losing it
    if not args.no_e2e and not w.offload:
        try:
            out["e2e"] = e2e_leg(b, min(args.steps, 10), world, dist, ms / args.steps)
        except Exception as exc:                      # e.g. pinned host memory not available
            out["e2e"] = {"value": None, "unit": UNIT, "error": f"{type(exc).__name__}: {exc}"[:300]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            out["cpu_baseline"] = cpu_baseline(w, args.cpu_sample_elems)
        except Exception as exc:
            out["cpu_baseline"] = {"value": None, "unit": UNIT, "kind": "oracle",
                                   "error": f"{type(exc).__name__}: {exc}"[:300]}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def e2e_leg(b: Bench, steps: int, world: int, dist, device_ms_per_step: float):
    """Same metric through the C ABI with host buffers: every step, for every bucket / unit,
    zero_step_host copies that call's contributions from pinned host memory into a device
    staging area (the next call's copies run while this call's step does), runs the step and
    copies the updated 16-bit parameters back into pinned host memory; (stage 3: the unit's
    all-gather first; with clipping, zero_grad_norm_host over every call before the steps;)
    zero_step_host_finish ends the step, waits for the copies and reads the step state.  Host gradients: two pinned sets of N_d buffers of the largest call's range,
    used by alternate calls (every byte crosses the host->device link every step; a set is
    far larger than the host CPU's caches).  The same steps with the library's serial schedule
    (ZERO_OPT_HOST_PIPELINE = 0: each call's copies, step and copy back one after another)
    show what the pipelining hides."""
    torch, Z, w = b.torch, b.Z, b.w
    g = b.g
    g.bind_host_staging()
    n_max = int(b.info.max_contrib_elems)
    host_sets = [[torch.empty(max(8, n_max), dtype=torch.int16, pin_memory=True)
                  for _ in range(w.n_d)] for _ in range(2)]
    # contents: the device gradients of the first call (the values do not change the speed)
    first = b.read_spans[0][0] if b.read_spans[0] else (0, 0, 0, 0)
    for hs in host_sets:
        for r in range(w.n_d):
            lo, hi, o, rel = first
            n = min(hi - lo, n_max - rel)
            if n > 0:
                hs[r][rel:rel + n].copy_(b.sets[0][r][o:o + n])
    host_out = torch.empty(max(8, b.set_elems), dtype=torch.int16, pin_memory=True)
    outs = []
    for ci in range(len(b.calls)):
        spans = b.read_spans[ci]
        a, e_, o, rel = spans[0] if spans else (0, 0, 0, 0)
        assert o - rel >= 0, "host results are laid out like the compact device sets"
        outs.append(host_out.data_ptr() + 2 * (o - rel))
    torch.cuda.synchronize()

    enqueue_s = [0.0]

    def one_step():
        t = time.perf_counter()
        if b.clip:                       # clipping: every call's norm pre-pass from host memory first
            for ci, (which, lo, hi) in enumerate(b.calls):
                g.grad_norm_host([t.data_ptr() for t in host_sets[ci % 2]], which)
        for ci, (which, lo, hi) in enumerate(b.calls):
            if w.stage == 3:
                g.gather(which, b.run.gather_buf)
                g.release(which)
            g.step_host([t.data_ptr() for t in host_sets[ci % 2]], which, b.hyper, outs[ci])
        enqueue_s[0] += time.perf_counter() - t
        return g.finish_host()             # waits for every copy; reads the step state back

    def timed(n):
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t = time.perf_counter()
        applied = 0
        for _ in range(n):
            applied += 1 - one_step().skipped
        el = time.perf_counter() - t
        if dist:
            el = max_over_ranks(el, dist)
        return el, applied

    one_step()                                            # warm-up (creates the copy streams)
    link_peak = h2d_copy_gbs()
    enqueue_s[0] = 0.0
    el, applied = timed(steps)
    enqueue_ms = 1e3 * enqueue_s[0] / steps
    h2d = Z.zero_get_option(g.plan, Z.ZERO_OPT_HOST_H2D_BYTES)
    d2h = Z.zero_get_option(g.plan, Z.ZERO_OPT_HOST_D2H_BYTES)
    g.set_option(Z.ZERO_OPT_HOST_PIPELINE, 0)
    n_serial = max(1, min(3, steps))
    el_serial, _ = timed(n_serial)
    g.set_option(Z.ZERO_OPT_HOST_PIPELINE, 1)
    ms = 1e3 * el / steps
    ms_serial = 1e3 * el_serial / n_serial
    hidden_ms = ms_serial - ms
    step_bytes = b.elems_per_step * b.bytes_per_elem
    hidden_frac = max(0.0, min(1.0, hidden_ms / device_ms_per_step)) if device_ms_per_step > 0 else 0.0
    return {"value": job_value(b.elems_per_step, applied, world, el), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h) + 96,
            "steps": steps,
            "api": ("zero_grad_norm_host / " if b.clip else "") + "zero_step_host / zero_step_host_finish",
            "host_link_gbs": round((h2d + d2h) / (ms / 1e3) / 1e9, 1),
            # host->device bytes per second against one plain pinned 1 GB copy in this run
            "h2d_gbs": round(h2d / (ms / 1e3) / 1e9, 1), "h2d_copy_peak_gbs": round(link_peak, 1),
            "h2d_frac": round(h2d / (ms / 1e3) / 1e9 / link_peak, 4),
            "host_enqueue_ms_per_step": round(enqueue_ms, 3),
            "overlap": {"pipelined_ms_per_step": round(ms, 3),
                        "serial_ms_per_step": round(ms_serial, 3),
                        "hidden_ms_per_step": round(hidden_ms, 3),
                        "device_step_ms": round(device_ms_per_step, 3),
                        "device_step_hidden_fraction": round(hidden_frac, 4),
                        "device_step_bytes_hidden": int(hidden_frac * step_bytes)}}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample_run(w, sample_elems: int, steps: int, warmup: int = 0):
    """Time the CPU oracle (single thread) on the first `sample_elems` flat elements."""
    import numpy as np
    import oracle                      # the CPU baseline legs alone load the oracle
    import synth
    from synth.fill import fill_host
    L = oracle.Layout(w.sizes, w.n_d, w.unit_first or None)
    units = [tuple(int(x) for x in u) for u in L.units]
    n = min(sample_elems, L.total_pad)
    p = oracle.widen16(fill_host(synth.param_stream(w), units, 0, n), w.dtype).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    out16 = np.zeros(n, np.uint16)
    sc = oracle.ScalerState(w.scaler)
    times = []
    for k in range(1, warmup + steps + 1):
        c = [fill_host(synth.grad_stream(w, k, r), units, 0, n) for r in range(w.n_d)]
        t = time.perf_counter()
        k9 = oracle.consts(w.hyper, sc.t + 1, sc.scale, w.n_d)
        g, flag = oracle.reduce(c, w.dtype, float(k9[8]))
        if flag:
            oracle.recast(p, w.dtype, out16)
        else:
            oracle.adamw(g, p, m, v, k9, w.dtype, out16)
        sc.update(flag)
        if k > warmup:
            times.append(time.perf_counter() - t)
    return n, times


def h2d_copy_gbs(n_bytes: int = 1 << 30, reps: int = 3) -> float:
    """Host->device copy rate (best of `reps`) of one pinned 1 GB buffer by the copy engine:
    the peak the end-to-end leg's host->device bytes are compared with."""
    import torch
    src = torch.ones(n_bytes // 2, dtype=torch.int16, pin_memory=True)
    dst = torch.empty(n_bytes // 2, dtype=torch.int16, device="cuda")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps + 1):                 # the first copy warms the path
        torch.cuda.synchronize()
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del src, dst
    return n_bytes / (best / 1e3) / 1e9


def host_copy_gbs(threads: int, n_bytes: int = 1 << 30, reps: int = 3) -> float:
    """Host memory copy bandwidth (read + write bytes / s, best of `reps`) of a 1 GB fp32 copy
    by torch's CPU kernels on `threads` threads."""
    import time
    import torch
    old = torch.get_num_threads()
    torch.set_num_threads(threads)
    try:
        src = torch.ones(n_bytes // 4, dtype=torch.float32)
        dst = torch.empty_like(src)
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            dst.copy_(src)
            best = min(best, time.perf_counter() - t0)
        return 2 * n_bytes / best / 1e9
    finally:
        torch.set_num_threads(old)


def cpu_baseline(w, sample_elems: int):
    n, times = oracle_sample_run(w, sample_elems, 2)
    return {"value": n * len(times) / sum(times), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {n} flat elements of {w.name}, {len(times)} steps, single-threaded "
                      f"oracle (reduce over {w.n_d} ranks + AdamW + cast), input generation excluded",
            "host_cpus": os.cpu_count()}


def reference_arm(args, world, rank):
    if rank != 0:
        return
    from synth import workloads as W
    w = W.workload(args.config)
    n, times = oracle_sample_run(w, args.cpu_sample_elems, max(1, args.steps), args.warmup)
    total = sum(times)
    value = n * len(times) / total
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic",
           "config": {"workload": w.name, "workload_index": args.config, "n_d": w.n_d,
                      "stage": w.stage, "phi": w.phi, "sample_elems": n},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": f"first {n} flat elements per step, single-threaded"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return
    gpu_arm(args, world, rank, local)


if __name__ == "__main__":
    main()
