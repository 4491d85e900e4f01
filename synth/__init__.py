"""Seeded synthetic inputs for the fused MoE expert block.

This module only draws inputs. It holds none of the block's arithmetic
(no quantisation, no GEMM, no SwiGLU, no combine), so both the CPU oracle
and the CUDA path can consume what it produces without sharing any of the
method's code.

Every random number comes from one counter-based generator: the 32-bit
MurmurHash3 finaliser ("fmix32", Appleby 2011) applied to a key built from
(seed, stream, counter), written in C (synth_gen.c) and run on the host.
The big INT8 weight tensors are drawn by position, so the oracle can redraw
only the experts it needs.  Floating inputs (x, scales) are drawn in float64
and rounded once.

Workloads follow the expert block's five synthetic configurations:

  tiny      bs 8,    h 256,  E 8,   topk 2, I 128,  no shared, no mask
  decode8   bs 8,    h 4096, E 256, topk 8, I 2048, shared expert
  decode64  bs 64,   same shapes, Zipf(1.2) routing, 25 % tokens masked,
            per-channel smooth scales U(0.8, 1.2)
  mid512    bs 512,  uniform routing, shared expert
  prefill   bs 4096, balanced routing (every expert gets 128 rows), shared

x ~ N(0,1) in bf16; weights uniform integers in [-127, 127]; per output
channel scales U(0.5, 1.5) / (127 sqrt(K)); expert_scales = softmax of topk
N(0,1) logits.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
from typing import Dict, Optional

import torch

# ---------------------------------------------------------------------------
# counter-based generator (C, synth_gen.c)
# ---------------------------------------------------------------------------
# stream ids: one per drawn quantity
S_X1, S_X2 = 1, 2
S_IDS, S_LOGITS1, S_LOGITS2 = 3, 4, 5
S_W1, S_W1S, S_W2, S_W2S = 6, 7, 8, 9
S_SMOOTH, S_SSMOOTH, S_MASK, S_PERM, S_TOKPERM = 10, 11, 12, 13, 14
S_ZIPF = 15

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.c")
_SO = os.path.join(_HERE, "_synth.so")
_lib = None


def build() -> str:
    """Compile the generator (gcc) next to its source if missing or stale."""
    if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               _SRC, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


def _get():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_hash_range.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint64,
                                         ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_hash_range.restype = None
        lib.synth_int8_uniform.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint64,
                                           ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int]
        lib.synth_int8_uniform.restype = ctypes.c_int
        _lib = lib
    return _lib


def hash_range(seed: int, stream: int, start: int, count: int) -> torch.Tensor:
    """hash(seed, stream, start + i) for i < count, as int64 values in [0, 2**32)."""
    out = torch.empty(count, dtype=torch.int32)
    if count:
        _get().synth_hash_range(seed, stream, start, count, out.data_ptr())
    return out.to(torch.int64) & 0xFFFFFFFF


def uniform01(seed: int, stream: int, start: int, count: int) -> torch.Tensor:
    """U[0,1) as float64 with 24 random bits (exact in float32)."""
    return (hash_range(seed, stream, start, count) >> 8).to(torch.float64) * (1.0 / (1 << 24))


def normal(seed: int, stream_a: int, stream_b: int, start: int, count: int) -> torch.Tensor:
    """N(0,1) by Box-Muller in float64 from two independent uniforms."""
    u1 = ((hash_range(seed, stream_a, start, count) >> 8).to(torch.float64) + 1.0) * (1.0 / (1 << 24))
    u2 = uniform01(seed, stream_b, start, count)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def int8_uniform(seed: int, stream: int, start: int, count: int, device="cpu",
                 threads: Optional[int] = None) -> torch.Tensor:
    """`count` integers uniform in [-127, 127] for flat positions start..start+count-1.

    Drawn on the host (multi-threaded C) and copied to `device` if needed."""
    if threads is None:
        threads = min(64, os.cpu_count() or 1)
    host = torch.empty(count, dtype=torch.int8)
    if count:
        _get().synth_int8_uniform(seed, stream, start, count, host.data_ptr(), threads)
    if str(device) == "cpu":
        return host
    return host.to(device)


def permutation(seed: int, stream: int, n: int) -> torch.Tensor:
    """Seeded permutation of range(n) (argsort of hashed keys, ties by index)."""
    keys = hash_range(seed, stream, 0, n)
    return torch.sort(keys * n + torch.arange(n, dtype=torch.int64), stable=True).indices


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    bs: int
    hidden: int
    num_experts: int
    topk: int
    inter: int
    has_shared: bool
    routing: str = "uniform"          # uniform | zipf | balanced
    masked_fraction: float = 0.0      # exact fraction of tokens set inactive
    smooth: bool = False              # expert_smooth_scales U(0.8, 1.2)
    share_smooth: bool = False        # share_smooth_scales U(0.8, 1.2)
    seed: int = 1000
    act_dtype: str = "bf16"           # x (and the outputs): bf16 | fp16
    scale_dtype: str = "f32"          # routed weight scales: f32 | bf16 | fp16
    smooth_per_expert: bool = False   # expert_smooth_scales [E, h] instead of [h]


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 8, 256, 8, 2, 128, False, seed=1000),
    "decode8": Workload("decode8", 8, 4096, 256, 8, 2048, True, seed=1001),
    "decode64": Workload("decode64", 64, 4096, 256, 8, 2048, True, routing="zipf",
                         masked_fraction=0.25, smooth=True, seed=1002),
    "mid512": Workload("mid512", 512, 4096, 256, 8, 2048, True, seed=1003),
    "prefill": Workload("prefill", 4096, 4096, 256, 8, 2048, True, routing="balanced", seed=1004),
}


@dataclasses.dataclass
class MoeInputs:
    """One batch of inputs. Small tensors live on the CPU; the weights live on
    `weight_device`.  Shapes follow the operator signature:
    x [bs,h] bf16, expert_ids [bs,k] int32, expert_scales [bs,k] f32,
    w1 [E,2I,h] int8 (rows 0..I-1 gate, I..2I-1 up), w1_scale [E,2I] f32,
    w2 [E,h,I] int8, w2_scale [E,h] f32, shared weights without the E axis,
    smooth scales [h] f32, x_active_mask [bs] bool.  Signature variants: x
    fp16; routed weight scales bf16 / fp16 (the f32 draw cast once);
    expert smooth scales [E, h]."""
    wl: Workload
    x: torch.Tensor
    expert_ids: torch.Tensor
    expert_scales: torch.Tensor
    w1: Optional[torch.Tensor]
    w1_scale: torch.Tensor
    w2: Optional[torch.Tensor]
    w2_scale: torch.Tensor
    share_w1: Optional[torch.Tensor] = None
    share_w1_scale: Optional[torch.Tensor] = None
    share_w2: Optional[torch.Tensor] = None
    share_w2_scale: Optional[torch.Tensor] = None
    smooth: Optional[torch.Tensor] = None
    share_smooth: Optional[torch.Tensor] = None
    mask: Optional[torch.Tensor] = None

    # host-side redraw of one expert's weights (expert == E means the shared expert)
    def expert_w1(self, e: int) -> torch.Tensor:
        return draw_w1(self.wl, e, "cpu")

    def expert_w2(self, e: int) -> torch.Tensor:
        return draw_w2(self.wl, e, "cpu")


def _wl_seed(wl: Workload) -> int:
    return wl.seed


def draw_w1(wl: Workload, e: int, device="cpu") -> torch.Tensor:
    """W1 of expert e ([2I, h]); e == E draws the shared expert."""
    n = 2 * wl.inter * wl.hidden
    return int8_uniform(_wl_seed(wl), S_W1, e * n, n, device).view(2 * wl.inter, wl.hidden)


def draw_w2(wl: Workload, e: int, device="cpu") -> torch.Tensor:
    """W2 of expert e ([h, I]); e == E draws the shared expert."""
    n = wl.hidden * wl.inter
    return int8_uniform(_wl_seed(wl), S_W2, e * n, n, device).view(wl.hidden, wl.inter)


def draw_all_w1(wl: Workload, device="cpu") -> torch.Tensor:
    n = 2 * wl.inter * wl.hidden
    return int8_uniform(_wl_seed(wl), S_W1, 0, wl.num_experts * n, device).view(
        wl.num_experts, 2 * wl.inter, wl.hidden)


def draw_all_w2(wl: Workload, device="cpu") -> torch.Tensor:
    n = wl.hidden * wl.inter
    return int8_uniform(_wl_seed(wl), S_W2, 0, wl.num_experts * n, device).view(
        wl.num_experts, wl.hidden, wl.inter)


def _channel_scales(seed: int, stream: int, rows: int, cols: int, k: int, start: int = 0) -> torch.Tensor:
    u = uniform01(seed, stream, start, rows * cols)
    c = 1.0 / (127.0 * math.sqrt(k))
    return ((0.5 + u) * c).to(torch.float32).view(rows, cols)


def _route_uniform(wl: Workload) -> torch.Tensor:
    E, k, bs = wl.num_experts, wl.topk, wl.bs
    keys = hash_range(wl.seed, S_IDS, 0, bs * E).view(bs, E)
    order = torch.sort(keys * E + torch.arange(E, dtype=torch.int64), dim=1, stable=True).indices
    return order[:, :k].to(torch.int32).contiguous()


def _route_zipf(wl: Workload, s: float = 1.2) -> torch.Tensor:
    """topk distinct ranks per token drawn without replacement with P(rank r) ~ r**-s
    (Efraimidis-Spirakis keys), then mapped to experts by a seeded permutation."""
    E, k, bs = wl.num_experts, wl.topk, wl.bs
    p = torch.arange(1, E + 1, dtype=torch.float64) ** (-s)
    p = p / p.sum()
    u = uniform01(wl.seed, S_ZIPF, 0, bs * E).view(bs, E)
    keys = torch.log(u + 2.0 ** -30) / p          # larger is better; log(u)/p = log(u**(1/p))
    ranks = torch.topk(keys, k, dim=1, largest=True, sorted=True).indices
    perm = permutation(wl.seed, S_PERM, E)
    return perm[ranks].to(torch.int32).contiguous()


def _route_balanced(wl: Workload) -> torch.Tensor:
    """ids[t][j] = pi((k*t + j) mod E); tokens then shuffled. Each expert gets bs*k/E rows."""
    E, k, bs = wl.num_experts, wl.topk, wl.bs
    pi = permutation(wl.seed, S_PERM, E)
    t = torch.arange(bs, dtype=torch.int64).view(bs, 1)
    j = torch.arange(k, dtype=torch.int64).view(1, k)
    ids = pi[(k * t + j) % E]
    sigma = permutation(wl.seed, S_TOKPERM, bs)
    return ids[sigma].to(torch.int32).contiguous()


def make_inputs(wl: Workload, weight_device="cpu", with_weights: bool = True) -> MoeInputs:
    """Draw every input of `wl`.  With with_weights=False the big INT8 weight tensors
    are left out (w1 = w2 = None); redraw them per expert with draw_w1/draw_w2."""
    seed, bs, h, E, k, I = wl.seed, wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    act = {"bf16": torch.bfloat16, "fp16": torch.float16}[wl.act_dtype]
    x = normal(seed, S_X1, S_X2, 0, bs * h).view(bs, h).to(act)

    if wl.routing == "uniform":
        ids = _route_uniform(wl)
    elif wl.routing == "zipf":
        ids = _route_zipf(wl)
    elif wl.routing == "balanced":
        ids = _route_balanced(wl)
    else:
        raise ValueError(wl.routing)

    logits = normal(seed, S_LOGITS1, S_LOGITS2, 0, bs * k).view(bs, k)
    scales = torch.softmax(logits, dim=1).to(torch.float32).contiguous()

    sdt = {"f32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[wl.scale_dtype]
    w1s = _channel_scales(seed, S_W1S, E, 2 * I, h).to(sdt)
    w2s = _channel_scales(seed, S_W2S, E, h, I).to(sdt)
    w1 = draw_all_w1(wl, weight_device) if with_weights else None
    w2 = draw_all_w2(wl, weight_device) if with_weights else None

    inp = MoeInputs(wl, x, ids, scales, w1, w1s, w2, w2s)
    if wl.has_shared:
        inp.share_w1 = draw_w1(wl, E, weight_device) if with_weights else None
        inp.share_w2 = draw_w2(wl, E, weight_device) if with_weights else None
        inp.share_w1_scale = _channel_scales(seed, S_W1S, 1, 2 * I, h, start=E * 2 * I).view(2 * I)
        inp.share_w2_scale = _channel_scales(seed, S_W2S, 1, h, I, start=E * h).view(h)
    if wl.smooth:
        n = E * h if wl.smooth_per_expert else h
        sm = (0.8 + 0.4 * uniform01(seed, S_SMOOTH, 0, n)).to(torch.float32)
        inp.smooth = sm.view(E, h) if wl.smooth_per_expert else sm
    if wl.share_smooth:
        inp.share_smooth = (0.8 + 0.4 * uniform01(seed, S_SSMOOTH, 0, h)).to(torch.float32)
    if wl.masked_fraction > 0:
        n_off = int(round(wl.masked_fraction * bs))
        perm = permutation(seed, S_MASK, bs)
        mask = torch.ones(bs, dtype=torch.bool)
        mask[perm[:n_off]] = False
        inp.mask = mask
    return inp


def custom(name="custom", bs=8, hidden=256, num_experts=8, topk=2, inter=128, has_shared=False,
           routing="uniform", masked_fraction=0.0, smooth=False, share_smooth=False, seed=7,
           act_dtype="bf16", scale_dtype="f32", smooth_per_expert=False) -> Workload:
    """A workload with arbitrary shapes (tests use these for ragged and edge cases)."""
    return Workload(name, bs, hidden, num_experts, topk, inter, has_shared, routing,
                    masked_fraction, smooth, share_smooth, seed, act_dtype, scale_dtype,
                    smooth_per_expert)


def touched_experts(ids: torch.Tensor, num_experts: int, mask: Optional[torch.Tensor] = None):
    """Sorted list of expert ids that at least one active (token, k) pair selects."""
    sel = ids
    if mask is not None:
        sel = ids[mask]
    v = sel.reshape(-1)
    v = v[(v >= 0) & (v < num_experts)]
    return sorted(set(int(a) for a in v.tolist()))
