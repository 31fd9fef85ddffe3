"""An emulated data-parallel group on one GPU.

The N_d ranks of the group live in one GPU's HBM: each bound rank owns its fp32
master/m/v shard (a ping-pong pair each), stage 3 ranks own a 16-bit parameter
shard, and stages 1/2 share one flat 16-bit parameter buffer (every replica is
identical).  This module only allocates those buffers with torch and forwards
them to the C ABI; every step of the optimizer runs in libzero's kernels.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import torch

from . import (ZERO_BF16, zero_set_option, ZERO_TABLE_PARAM_CHUNKS, ZERO_TABLE_STATE_LAYOUT, ZERO_TABLE_UNITS,
               zero_bind, zero_bind_offload, zero_bind_peer, zero_offload_finish,
               zero_offload_step, zero_plan_create_per_param,
               zero_gather_layer, zero_plan_create, zero_plan_destroy, zero_plan_info,
               zero_grad_norm, zero_plan_tables, zero_rank_state_elems, zero_read_state,
               zero_release_layer,
               zero_set_scaler, zero_step, zero_step_finish,
               zero_bind_host_staging, zero_step_host, zero_step_host_finish, zero_grad_norm_host,
               zero_step_gather_next)


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class EmulatedGroup:
    """Plan + device buffers of N_d emulated ranks (only `bound_ranks` carry optimizer state)."""

    def __init__(self, sizes: Sequence[int], n_d: int, stage: int, bucket_elems: int = 0,
                 unit_first: Optional[Sequence[int]] = None, dtype16: int = ZERO_BF16,
                 bound_ranks: Optional[Sequence[int]] = None, device: str = "cuda",
                 dim0: Optional[Sequence[int]] = None, offload: bool = False,
                 offload_threads: int = 0):
        """dim0 given: FSDP-2 per-parameter sharding (stage-3 semantics) instead of flat units.
        offload: ZeRO-Offload -- the bound ranks' fp32 state lives in (pinned) host memory and is
        updated by `offload_threads` CPU threads (default: all CPUs)."""
        import os
        self.device = torch.device(device)
        self.offload = offload
        self.offload_threads = offload_threads or (os.cpu_count() or 1)
        self.n_d, self.dtype16 = n_d, dtype16
        self.per_param = dim0 is not None
        self.stage = 3 if self.per_param else stage
        if self.per_param:
            self.plan = zero_plan_create_per_param(list(sizes), list(dim0), n_d,
                                                   list(unit_first) if unit_first else None, dtype16)
        else:
            self.plan = zero_plan_create(list(sizes), n_d, stage, bucket_elems,
                                         list(unit_first) if unit_first else None, dtype16)
        stage = self.stage
        self.info = zero_plan_info(self.plan)
        self.units = zero_plan_tables(self.plan, ZERO_TABLE_UNITS)
        self.phys_off: Dict[int, List[int]] = {}
        self.chunks = []
        if self.per_param:
            # rank, unit, tensor, row0, rows, cols, c_rows, contrib_off, state_off, phys_off
            self.chunks = zero_plan_tables(self.plan, ZERO_TABLE_PARAM_CHUNKS)
        else:
            for r, u, off, _n in zero_plan_tables(self.plan, ZERO_TABLE_STATE_LAYOUT):
                self.phys_off.setdefault(r, []).append(off)
        self.bound = list(bound_ranks) if bound_ranks is not None else list(range(n_d))
        self.state: Dict[int, Dict[str, List[torch.Tensor]]] = {}
        self.shard16: Dict[int, torch.Tensor] = {}
        self.workspace = torch.zeros(int(self.info.workspace_bytes) // 4, dtype=torch.int32,
                                     device=self.device)
        self.full16 = None
        if stage != 3:
            self.full16 = torch.zeros(int(self.info.phi_pad), dtype=torch.int16, device=self.device)
        self.grad_host: Dict[int, torch.Tensor] = {}
        self.param16_host: Dict[int, torch.Tensor] = {}
        for r in self.bound:
            n = zero_rank_state_elems(self.plan, r)
            if offload:
                st = {k: [torch.zeros(n, dtype=torch.float32, pin_memory=True)]
                      for k in ("master", "m", "v")}
                self.state[r] = st
                self.grad_host[r] = torch.zeros(n, dtype=torch.float32, pin_memory=True)
                self.param16_host[r] = torch.zeros(n, dtype=torch.int16, pin_memory=True)
                sh = None
                if stage == 3:
                    sh = torch.zeros(n, dtype=torch.int16, device=self.device)
                    self.shard16[r] = sh
                zero_bind_offload(self.plan, r, st["master"][0].data_ptr(), st["m"][0].data_ptr(),
                                  st["v"][0].data_ptr(), self.grad_host[r].data_ptr(),
                                  self.param16_host[r].data_ptr(),
                                  sh.data_ptr() if sh is not None else None,
                                  self.full16.data_ptr() if self.full16 is not None else None,
                                  self.workspace.data_ptr())
                continue
            st = {k: [torch.zeros(n, dtype=torch.float32, device=self.device) for _ in range(2)]
                  for k in ("master", "m", "v")}
            self.state[r] = st
            sh = None
            if stage == 3:
                sh = torch.zeros(n, dtype=torch.int16, device=self.device)
                self.shard16[r] = sh
            zero_bind(self.plan, r, [t.data_ptr() for t in st["master"]],
                      [t.data_ptr() for t in st["m"]], [t.data_ptr() for t in st["v"]],
                      sh.data_ptr() if sh is not None else None,
                      self.full16.data_ptr() if self.full16 is not None else None,
                      self.workspace.data_ptr())

    # ------------------------------------------------------------------ layout helpers
    def shard_slices(self, rank: int):
        """(unit, physical offset, length, unit base, unit shard size) of the rank's shard."""
        out = []
        for u, (first, count, numel, numel_pad, shard, base, shard_base) in enumerate(self.units):
            out.append((u, self.phys_off[rank][u], shard, base, shard))
        return out

    def bind_peer_shard(self, rank: int) -> torch.Tensor:
        """Stage 3: allocate and register the 16-bit shard of a rank without local state."""
        n = zero_rank_state_elems(self.plan, rank)
        sh = torch.zeros(n, dtype=torch.int16, device=self.device)
        zero_bind_peer(self.plan, rank, sh.data_ptr())
        self.shard16[rank] = sh
        return sh

    def step_state(self, stream=None):
        """Device-resident step state (synchronises the stream)."""
        return zero_read_state(self.plan, _stream_handle(stream))

    def current(self) -> int:
        return self.step_state().current

    def t(self) -> int:
        return self.step_state().t

    def set_scaler(self, scaler, stream=None) -> None:
        zero_set_scaler(self.plan, scaler, _stream_handle(stream))

    def set_option(self, option: int, value: int) -> None:
        zero_set_option(self.plan, option, value)

    def state_tensor(self, rank: int, name: str) -> torch.Tensor:
        if self.offload:                       # updated in place on the host
            return self.state[rank][name][0]
        return self.state[rank][name][self.current()]

    def rank_chunks(self, rank: int):
        """Per-parameter plans: the rank's chunks (rank, unit, tensor, row0, rows, cols, c_rows,
        contrib_off, state_off, phys_off)."""
        return [c for c in self.chunks if c[0] == rank]

    def logical(self, rank: int, phys: torch.Tensor) -> torch.Tensor:
        """Gather a rank's buffer from the physical layout into logical shard order."""
        if self.per_param:
            parts = [phys[c[9]:c[9] + c[6] * c[5]] for c in self.rank_chunks(rank)]
            return torch.cat(parts) if parts else phys[:0]
        parts = [phys[off:off + n] for (_u, off, n, _b, _s) in self.shard_slices(rank)]
        return torch.cat(parts) if parts else phys[:0]

    # ------------------------------------------------------------------ the step
    def step(self, contribs: Sequence[int], which: int, hyper, stream=None) -> None:
        if self.offload:
            zero_offload_step(self.plan, list(contribs), which, hyper, _stream_handle(stream))
            return
        zero_step(self.plan, list(contribs), which, hyper, _stream_handle(stream))

    def bind_host_staging(self) -> None:
        """Allocate and bind the two device staging areas of the host-buffer path."""
        n = int(self.info.host_staging_bytes)
        self.host_staging = [torch.empty(max(16, n), dtype=torch.uint8, device=self.device)
                             for _ in range(2)]
        zero_bind_host_staging(self.plan, [t.data_ptr() for t in self.host_staging], max(16, n))

    def step_host(self, host_contribs: Sequence[int], which: int, hyper, host_out16: int,
                  stream=None) -> None:
        """zero_step with the contributions and the 16-bit result in pinned host memory."""
        zero_step_host(self.plan, list(host_contribs), which, hyper, host_out16,
                       _stream_handle(stream))

    def grad_norm_host(self, host_contribs: Sequence[int], which: int, stream=None) -> None:
        """Gradient-norm pre-pass of one bucket/unit fed from pinned host memory."""
        zero_grad_norm_host(self.plan, list(host_contribs), which, _stream_handle(stream))

    def finish_host(self, stream=None):
        """End a step with host-buffer calls (synchronises); returns the step state."""
        return zero_step_host_finish(self.plan, _stream_handle(stream))

    def grad_norm(self, contribs: Sequence[int], which: int, stream=None) -> None:
        """Gradient-norm pre-pass of one bucket/unit (needed before a clipping step)."""
        zero_grad_norm(self.plan, list(contribs), which, _stream_handle(stream))

    def finish(self, stream=None, wait: bool = True):
        """Commit the step on the device; wait=True also returns the read-back state."""
        if self.offload:
            return zero_offload_finish(self.plan, self.offload_threads, _stream_handle(stream), wait)
        return zero_step_finish(self.plan, _stream_handle(stream), wait)

    def step_gather_next(self, contribs: Sequence[int], unit: int, hyper, next_unit: int,
                         dst: torch.Tensor, stream=None) -> None:
        """Step of `unit` with the all-gather of `next_unit` into dst in the same launch."""
        zero_step_gather_next(self.plan, list(contribs), unit, hyper, next_unit, dst.data_ptr(),
                              _stream_handle(stream))

    def gather(self, unit: int, dst: torch.Tensor, stream=None) -> None:
        zero_gather_layer(self.plan, unit, dst.data_ptr(), _stream_handle(stream))

    def release(self, unit: int) -> None:
        zero_release_layer(self.plan, unit)

    def close(self) -> None:
        if self.plan:
            zero_plan_destroy(self.plan)
            self.plan = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
