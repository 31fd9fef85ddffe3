"""Synthetic workloads of the sharded mixed-precision AdamW step.

Each workload fixes the tensor-size list of a model shape (no weights: shapes
only), the data-parallel degree N_d, the ZeRO stage, the bucket size, the FSDP
unit boundaries (stage 3), the 16-bit dtype, the number of steps, the AdamW
hyperparameters and the recipe of the synthetic inputs.  Nothing here computes
any part of the step itself.

Recipes (value distributions) follow the workload descriptions this project is
measured on:
  * parameters ~ N(0, 0.02) in 16-bit; fp32 master = exact widening; m = v = 0;
  * gradient contributions ~ N(0, 1e-2), one independent stream per
    (step, rank); optional 1 % outliers x100; optional planted +inf.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

SEED = 0
BF16 = 0
FP16 = 1

KIND_PARAM = 1
KIND_GRAD = 2
KIND_SIZES = 3

INF16 = {BF16: 0x7F80, FP16: 0x7C00}


@dataclasses.dataclass(frozen=True)
class Hyper:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 0.0       # > 0: clip by the global gradient norm
    report_norm: bool = False        # compute the global gradient norm in the fused pass


@dataclasses.dataclass(frozen=True)
class Scaler:
    """Dynamic loss scale: skip + back off on inf/nan, grow after a clean run."""
    init_scale: float = 65536.0
    growth_factor: float = 2.0
    backoff_factor: float = 0.5
    growth_interval: int = 1000
    min_scale: float = 1.0


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int                      # workload id (keys the generator streams)
    name: str
    sizes: Tuple[int, ...]        # tensor sizes (elements), in flattening order
    n_d: int                      # data-parallel degree (emulated ranks)
    stage: int                    # 1, 2, 3
    bucket_elems: int             # 0 = one bucket over the whole flat buffer
    unit_first: Tuple[int, ...]   # first tensor of each FSDP unit (stage 3); () = one unit
    dtype: int                    # BF16 or FP16
    steps: int
    hyper: Hyper
    scaler: Optional[Scaler]      # None: loss scale 1, no dynamic scaling
    param_sigma: float = 0.02
    grad_sigma: float = 1e-2
    outliers: bool = False
    inject: Optional[Tuple[int, int, int]] = None   # (step 1-based, rank, flat index) of a +inf
    bound_ranks: Optional[Tuple[int, ...]] = None   # ranks whose shard is updated; None = all
    dim0: Optional[Tuple[int, ...]] = None          # leading dimension of every tensor
    per_param: bool = False                         # FSDP-2 per-parameter (dim-0) sharding
    offload: bool = False                           # ZeRO-Offload: fp32 state on the host CPU

    @property
    def phi(self) -> int:
        return sum(self.sizes)

    def units(self) -> List[Tuple[int, int]]:
        """(first tensor, tensor count) of each unit."""
        firsts = list(self.unit_first) if self.unit_first else [0]
        ends = firsts[1:] + [len(self.sizes)]
        return [(f, e - f) for f, e in zip(firsts, ends)]

    def ranks(self) -> Tuple[int, ...]:
        return self.bound_ranks if self.bound_ranks is not None else tuple(range(self.n_d))


def gpt2_block(d: int, ffn: int) -> List[int]:
    """GPT-2 block: ln_1 w,b; attn c_attn w,b; attn c_proj w,b; ln_2 w,b; mlp c_fc w,b; mlp c_proj w,b."""
    return [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * ffn, ffn, ffn * d, d]


def gpt_sizes(vocab: int, ctx: int, d: int, ffn: int, layers: int) -> Tuple[List[int], List[int]]:
    """GPT-2-style tensor list with a tied head: wte, wpe, blocks, ln_f.

    Returns (sizes, unit_first) with units = {embeddings}, one per block, {ln_f}.
    """
    sizes = [vocab * d, ctx * d]
    unit_first = [0]
    for _ in range(layers):
        unit_first.append(len(sizes))
        sizes += gpt2_block(d, ffn)
    unit_first.append(len(sizes))
    sizes += [d, d]
    return sizes, unit_first


def gpt_dim0(vocab: int, ctx: int, d: int, ffn: int, layers: int) -> List[int]:
    """Leading dimensions of gpt_sizes' tensors (Conv1D weights are stored (in, out))."""
    dims = [vocab, ctx]
    for _ in range(layers):
        dims += [d, d, d, 3 * d, d, d, d, d, d, ffn, ffn, d]
    return dims + [d, d]


def llama_dim0(vocab: int, d: int, ffn: int, layers: int) -> List[int]:
    """Leading dimensions of llama_sizes' tensors (Linear weights are stored (out, in))."""
    dims = [vocab]
    for _ in range(layers):
        dims += [d, d, d, d, d, d, ffn, ffn, d]
    return dims + [d, vocab]


def unit_slice(w: "Workload", u: int, n_units: int = 1) -> "Workload":
    """Stage 3: the same workload restricted to the tensors of units u .. u + n_units - 1, e.g.
    to profile one or two units' kernels with a few GB on the device."""
    if w.stage != 3:
        raise ValueError("unit_slice: stage-3 workloads only")
    units = w.units()[u:u + n_units]
    if not units or n_units < 1:
        raise ValueError("unit_slice: no such units")
    first = units[0][0]
    last = units[-1][0] + units[-1][1]
    firsts = tuple(f - first for f, _ in units)
    label = f"unit {u} only" if n_units == 1 else f"units {u}..{u + n_units - 1} only"
    return dataclasses.replace(
        w, name=f"{w.name}, {label}", sizes=w.sizes[first:last], unit_first=firsts,
        dim0=w.dim0[first:last] if w.dim0 else None, inject=None)


def per_param_variant(w: "Workload") -> "Workload":
    """The same workload under FSDP-2 per-parameter sharding (stage-3 semantics)."""
    assert w.dim0 is not None
    units = w.unit_first if w.unit_first else (0,)
    return dataclasses.replace(w, wid=w.wid + 100, name=w.name + "_per_param", stage=3,
                               bucket_elems=0, unit_first=units, per_param=True)


def llama_sizes(vocab: int, d: int, ffn: int, layers: int) -> Tuple[List[int], List[int]]:
    """Llama-style tensor list, untied head: embed, blocks, final norm + lm_head.

    Block order: input norm, q, k, v, o, post-attention norm, gate, up, down.
    Units = {embed}, one per block, {final norm, lm_head}.
    """
    sizes = [vocab * d]
    unit_first = [0]
    for _ in range(layers):
        unit_first.append(len(sizes))
        sizes += [d, d * d, d * d, d * d, d * d, d, d * ffn, d * ffn, ffn * d]
    unit_first.append(len(sizes))
    sizes += [d, vocab * d]
    return sizes, unit_first


def loguniform_sizes(n: int, lo_log2: int = 0, hi_log2: int = 16, wid: int = 1) -> List[int]:
    """n tensor sizes, log-uniform in [1, 65536]: floor(2^(16 u)), u uniform in [0, 1).

    u comes from the top 53 bits of splitmix64 over a counter, keyed like the
    other streams; the result is clamped to [1, 2^16].
    """
    from . import hash64, stream_key
    key = stream_key(SEED, wid, KIND_SIZES, 0, 0)
    out = []
    span = hi_log2 - lo_log2
    for t in range(n):
        u = (hash64((key + t) & 0xFFFFFFFFFFFFFFFF) >> 11) / float(1 << 53)
        s = int(math.floor(2.0 ** (lo_log2 + span * u)))
        out.append(min(max(s, 1), 1 << hi_log2))
    return out


def _cfg0() -> Workload:
    return Workload(wid=0, name="zero1_flat_phi2^20_nd4_bf16", sizes=(1 << 20,), n_d=4, stage=1,
                    bucket_elems=0, unit_first=(), dtype=BF16, steps=3, hyper=Hyper(), scaler=None,
                    dim0=(1 << 20,))


def _cfg1() -> Workload:
    sizes = tuple(loguniform_sizes(10000, wid=1))
    return Workload(wid=1, name="zero2_ragged_10000tensors_nd7_bf16", sizes=sizes, n_d=7, stage=2,
                    bucket_elems=0, unit_first=(), dtype=BF16, steps=5, hyper=Hyper(), scaler=None,
                    dim0=sizes)


def _cfg2() -> Workload:
    sizes, _ = gpt_sizes(50257, 1024, 768, 3072, 12)
    phi = sum(sizes)
    return Workload(wid=2, name="zero2_bucketed_gpt2small_nd8_fp16", sizes=tuple(sizes), n_d=8,
                    stage=2, bucket_elems=25_000_000, unit_first=(), dtype=FP16, steps=10,
                    hyper=Hyper(), scaler=Scaler(), outliers=True, inject=(3, 0, phi // 2),
                    dim0=tuple(gpt_dim0(50257, 1024, 768, 3072, 12)))


def _cfg3() -> Workload:
    sizes, units = gpt_sizes(50257, 2048, 2048, 8192, 24)
    return Workload(wid=3, name="zero3_per_layer_gpt1.3b_nd16_bf16", sizes=tuple(sizes), n_d=16,
                    stage=3, bucket_elems=0, unit_first=tuple(units), dtype=BF16, steps=4,
                    hyper=Hyper(), scaler=None, dim0=tuple(gpt_dim0(50257, 2048, 2048, 8192, 24)))


def _cfg4() -> Workload:
    sizes, units = llama_sizes(32000, 4096, 11008, 32)
    return Workload(wid=4, name="zero3_one_rank_llama6.74b_nd8_bf16", sizes=tuple(sizes), n_d=8,
                    stage=3, bucket_elems=0, unit_first=tuple(units), dtype=BF16, steps=5,
                    hyper=Hyper(), scaler=None, bound_ranks=(0,),
                    dim0=tuple(llama_dim0(32000, 4096, 11008, 32)))


_BUILDERS = [_cfg0, _cfg1, _cfg2, _cfg3, _cfg4]
_CACHE = {}


def workload(i: int) -> Workload:
    if i not in _CACHE:
        _CACHE[i] = _BUILDERS[i]()
    return _CACHE[i]


N_WORKLOADS = len(_BUILDERS)
