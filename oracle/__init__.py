"""CPU oracle of the fused MoE expert block -- test infrastructure only.

`moe_oracle.c` is a plain, slow, step-by-step C restatement of the block as the
FusedDeepMoE analysis describes it (dispatch, per-token INT8 quant, grouped
GEMM1, dequant + SwiGLU, requant, grouped GEMM2, dequant to bf16, combine,
shared expert).  This wrapper only marshals arguments.  Only the tests, the
package smoke check and the benchmark's CPU-baseline leg may import it; the
CUDA product path never does, and the two share no code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# ORACLE_MUTANT_SRC / ORACLE_MUTANT_SO let the mutation test build a copy of
# the oracle with one planted mistake and check that the pins reject it.
_SRC = os.environ.get("ORACLE_MUTANT_SRC", os.path.join(_HERE, "moe_oracle.c"))
_SO = os.environ.get("ORACLE_MUTANT_SO", os.path.join(_HERE, "_moe_oracle.so"))
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fno-builtin-expf",
          "-shared", "-fPIC", "-pthread"]


def build() -> str:
    """Compile the oracle with gcc next to its source (if missing or stale)."""
    if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc"] + CFLAGS + [_SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


P = ctypes.c_void_p
I32 = ctypes.c_int32


class OracleArgs(ctypes.Structure):
    _fields_ = [("bs", I32), ("hidden", I32), ("num_experts", I32), ("topk", I32), ("inter", I32),
                ("has_shared", I32),
                ("x", P), ("expert_ids", P), ("expert_scales", P),
                ("w1", P), ("w1_scale", P), ("w2", P), ("w2_scale", P),
                ("share_w1", P), ("share_w1_scale", P), ("share_w2", P), ("share_w2_scale", P),
                ("smooth", P), ("share_smooth", P), ("mask", P), ("token_sample", P),
                ("threads", I32), ("fold_routing", I32),
                ("act_fp16", I32), ("scale_dtype", I32), ("smooth_per_expert", I32)]


class OracleOut(ctypes.Structure):
    _fields_ = [("output", P), ("share_output", P), ("expert_token_nums", P),
                ("offsets", P), ("row_of", P), ("tk_of_row", P),
                ("x_q", P), ("x_scale", P), ("xs_q", P), ("xs_scale", P),
                ("acc1", P), ("h_act", P), ("x2", P), ("s2", P), ("acc2", P), ("y2", P),
                ("share_acc1", P), ("share_h", P), ("share_x2", P), ("share_s2", P), ("share_acc2", P),
                ("skipped", I32), ("R", I32)]


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.oracle_forward.argtypes = [ctypes.POINTER(OracleArgs), ctypes.POINTER(OracleOut)]
        L.oracle_forward.restype = ctypes.c_int
        L.oracle_dispatch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P]
        L.oracle_dispatch.restype = ctypes.c_int
        L.oracle_quant_row.argtypes = [ctypes.c_int, P, P, P, P]
        L.oracle_quant_row.restype = None
        L.oracle_gemm_row.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P]
        L.oracle_gemm_row.restype = ctypes.c_int
        L.oracle_swiglu_row.argtypes = [ctypes.c_int, P, P, ctypes.c_float, P]
        L.oracle_swiglu_row.restype = None
        L.oracle_requant_row.argtypes = [ctypes.c_int, P, P, P]
        L.oracle_requant_row.restype = None
        L.oracle_dequant_bf16_row.argtypes = [ctypes.c_int, P, P, ctypes.c_float, P]
        L.oracle_dequant_bf16_row.restype = None
        L.oracle_combine_token.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P]
        L.oracle_combine_token.restype = None
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f32.restype = ctypes.c_float
        L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_f16.restype = ctypes.c_uint16
        L.oracle_sizeof_args.restype = ctypes.c_int
        L.oracle_sizeof_out.restype = ctypes.c_int
        assert L.oracle_sizeof_args() == ctypes.sizeof(OracleArgs)
        assert L.oracle_sizeof_out() == ctypes.sizeof(OracleOut)
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return t.data_ptr()


def _bits(x: torch.Tensor) -> torch.Tensor:
    """bf16 / fp16 tensor -> its raw 16-bit patterns (int16 view), contiguous CPU."""
    return x.detach().to("cpu").contiguous().view(torch.int16)


def _bf16(bits: torch.Tensor) -> torch.Tensor:
    return bits.view(torch.bfloat16)


def _act(bits: torch.Tensor, fp16: bool) -> torch.Tensor:
    return bits.view(torch.float16 if fp16 else torch.bfloat16)


_SCALE_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


def _scales(t: torch.Tensor) -> torch.Tensor:
    """Weight scales as stored: fp32 values, or the raw bits of bf16 / fp16."""
    t = t.detach().to("cpu").contiguous()
    return t if t.dtype == torch.float32 else t.view(torch.int16)


# ----------------------------------------------------------- step functions
def dispatch(ids: torch.Tensor, num_experts: int, mask: Optional[torch.Tensor] = None) -> Dict:
    """Counting sort of active (t, k) pairs: counts, offsets, row_of, tk_of_row."""
    ids = ids.to(torch.int32).contiguous()
    bs, k = ids.shape
    m = None if mask is None else mask.to(torch.uint8).contiguous()
    counts = torch.zeros(num_experts, dtype=torch.int32)
    offsets = torch.zeros(num_experts + 1, dtype=torch.int32)
    row_of = torch.full((bs * k,), -1, dtype=torch.int32)
    tk = torch.full((max(bs * k, 1),), -1, dtype=torch.int32)
    skipped = ctypes.c_int32(0)
    R = lib().oracle_dispatch(bs, k, num_experts, _ptr(ids), _ptr(m), _ptr(counts), _ptr(offsets),
                              _ptr(row_of), _ptr(tk), ctypes.addressof(skipped))
    return dict(counts=counts, offsets=offsets, row_of=row_of.view(bs, k), tk_of_row=tk[:R].clone(),
                R=R, skipped=skipped.value)


def quant_row(x_row: torch.Tensor, smooth: Optional[torch.Tensor] = None):
    """Per-token dynamic INT8 quant of one bf16 row -> (q int8 [h], scale float)."""
    xb = _bits(x_row.reshape(-1))
    h = xb.numel()
    q = torch.empty(h, dtype=torch.int8)
    s = ctypes.c_float(0.0)
    sm = None if smooth is None else smooth.to(torch.float32).contiguous()
    lib().oracle_quant_row(h, _ptr(xb), _ptr(sm), _ptr(q), ctypes.addressof(s))
    return q, s.value


def gemm_rows(a: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    """int32 acc[m][n] = sum_c a[m][c] * w[n][c] row by row (a [M,K] int8, w [N,K] int8)."""
    a = a.to(torch.int8).contiguous()
    w = w.to(torch.int8).contiguous()
    M, K = a.shape
    N = w.shape[0]
    out = torch.empty(M, N, dtype=torch.int32)
    for m in range(M):
        rc = lib().oracle_gemm_row(N, K, _ptr(a[m]), _ptr(w), _ptr(out[m]))
        if rc:
            raise ValueError("K too large for exact int32 accumulation")
    return out


def swiglu_row(acc1: torch.Tensor, w1s: torch.Tensor, x_scale: float) -> torch.Tensor:
    acc1 = acc1.to(torch.int32).contiguous()
    I = acc1.numel() // 2
    h = torch.empty(I, dtype=torch.float32)
    lib().oracle_swiglu_row(I, _ptr(acc1), _ptr(w1s.to(torch.float32).contiguous()), x_scale, _ptr(h))
    return h


def requant_row(h: torch.Tensor):
    h = h.to(torch.float32).contiguous()
    q = torch.empty(h.numel(), dtype=torch.int8)
    s = ctypes.c_float(0.0)
    lib().oracle_requant_row(h.numel(), _ptr(h), _ptr(q), ctypes.addressof(s))
    return q, s.value


def dequant_bf16_row(acc2: torch.Tensor, w2s: torch.Tensor, s2: float) -> torch.Tensor:
    acc2 = acc2.to(torch.int32).contiguous()
    y = torch.empty(acc2.numel(), dtype=torch.int16)
    lib().oracle_dequant_bf16_row(acc2.numel(), _ptr(acc2), _ptr(w2s.to(torch.float32).contiguous()),
                                  s2, _ptr(y))
    return _bf16(y)


def combine_token(rows: Sequence[Optional[torch.Tensor]], scales: torch.Tensor) -> torch.Tensor:
    keep = [_bits(r) if r is not None else None for r in rows]
    H = next(r.numel() for r in keep if r is not None)
    arr = (ctypes.c_void_p * len(keep))(*[r.data_ptr() if r is not None else None for r in keep])
    out = torch.empty(H, dtype=torch.int16)
    lib().oracle_combine_token(H, len(keep), ctypes.addressof(arr),
                               _ptr(scales.to(torch.float32).contiguous()), _ptr(out))
    return _bf16(out)


def bf16_round(v: float) -> int:
    return int(lib().oracle_f32_to_bf16(v)) & 0xFFFF


def f16_round(v: float) -> int:
    """fp16 code of v (round to nearest, ties to even)."""
    return int(lib().oracle_f32_to_f16(v)) & 0xFFFF


def f16_value(code: int) -> float:
    return float(lib().oracle_f16_to_f32(code & 0xFFFF))


# ------------------------------------------------------------- full block
def forward(inp, intermediates: bool = False, token_sample: Optional[torch.Tensor] = None,
            threads: Optional[int] = None, expert_weights=None, fold_routing: bool = False) -> Dict:
    """Run the whole block on the CPU.

    `inp` is a synth.MoeInputs (CPU tensors; weights may be absent, in which
    case the experts that active pairs select are redrawn one by one).
    `token_sample` (bool [bs]) restricts the GEMM work and the outputs to those
    tokens; dispatch still runs on every token.  `fold_routing` selects the
    mode in which each routed row's routing weight is folded into its GEMM2
    row scale and the combine is a plain sum.  The signature variants follow
    the inputs' own dtypes and shapes: fp16 x gives fp16 y2 and outputs,
    bf16 / fp16 routed weight scales are widened exactly, and a [E, h]
    smooth tensor makes the routed quant per row.  Returns a dict of tensors
    (outputs in x's dtype).
    """
    wl = inp.wl
    bs, h, E, K, I = wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    shared = bool(wl.has_shared)
    if threads is None:
        threads = int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1))
    x = _bits(inp.x)
    fp16 = inp.x.dtype == torch.float16
    if inp.w1_scale.dtype != inp.w2_scale.dtype:
        raise ValueError("routed weight scales must share one dtype")
    scale_dtype = _SCALE_DTYPES[inp.w1_scale.dtype]
    per_expert = inp.smooth is not None and inp.smooth.dim() == 2
    ids = inp.expert_ids.to(torch.int32).contiguous()
    sc = inp.expert_scales.to(torch.float32).contiguous()
    mask = None if inp.mask is None else inp.mask.to(torch.uint8).contiguous()
    samp = None if token_sample is None else token_sample.to(torch.uint8).contiguous()

    # experts whose weights are needed
    need = set()
    for t in range(bs):
        if mask is not None and not mask[t]:
            continue
        if samp is not None and not samp[t]:
            continue
        for e in ids[t].tolist():
            if 0 <= e < E:
                need.add(e)
    keep = []
    w1p = (ctypes.c_void_p * E)()
    w2p = (ctypes.c_void_p * E)()
    def host_weights(e):
        """Host copy of expert e's weights (e == E: the shared expert), never
        read back from a device: redrawn from the seeded generator instead."""
        if expert_weights is not None:
            return expert_weights(e)
        if e < E and inp.w1 is not None and inp.w1.device.type == "cpu":
            return inp.w1[e], inp.w2[e]
        if e == E and inp.share_w1 is not None and inp.share_w1.device.type == "cpu":
            return inp.share_w1, inp.share_w2
        return inp.expert_w1(e), inp.expert_w2(e)

    for e in sorted(need):
        a, b = host_weights(e)
        a = a.contiguous(); b = b.contiguous()
        keep += [a, b]
        w1p[e] = a.data_ptr(); w2p[e] = b.data_ptr()

    w1s = _scales(inp.w1_scale)
    w2s = _scales(inp.w2_scale)
    sw1 = sw2 = sw1s = sw2s = None
    if shared:
        sw1, sw2 = host_weights(E)
        sw1 = sw1.contiguous(); sw2 = sw2.contiguous()
        sw1s = inp.share_w1_scale.to(torch.float32).contiguous()
        sw2s = inp.share_w2_scale.to(torch.float32).contiguous()
    smooth = None if inp.smooth is None else inp.smooth.to(torch.float32).contiguous()
    ssmooth = None if inp.share_smooth is None else inp.share_smooth.to(torch.float32).contiguous()

    a = OracleArgs(bs, h, E, K, I, int(shared), _ptr(x), _ptr(ids), _ptr(sc),
                   ctypes.addressof(w1p), _ptr(w1s), ctypes.addressof(w2p), _ptr(w2s),
                   _ptr(sw1), _ptr(sw1s), _ptr(sw2), _ptr(sw2s), _ptr(smooth), _ptr(ssmooth),
                   _ptr(mask), _ptr(samp), threads, int(bool(fold_routing)),
                   int(fp16), scale_dtype, int(per_expert))

    res = {}
    res["output"] = torch.zeros(bs, h, dtype=torch.int16)
    res["share_output"] = torch.zeros(bs, h, dtype=torch.int16) if shared else None
    res["expert_token_nums"] = torch.zeros(E, dtype=torch.int32)
    o = OracleOut()
    o.output = _ptr(res["output"]); o.share_output = _ptr(res["share_output"])
    o.expert_token_nums = _ptr(res["expert_token_nums"])
    nrows = bs * K
    if intermediates:
        res["offsets"] = torch.zeros(E + 1, dtype=torch.int32)
        res["row_of"] = torch.full((bs, K), -1, dtype=torch.int32)
        res["tk_of_row"] = torch.full((max(nrows, 1),), -1, dtype=torch.int32)
        nq = nrows if per_expert else bs   # per routed row with [E, h] smooth scales
        res["x_q"] = torch.zeros(max(nq, 1), h, dtype=torch.int8)
        res["x_scale"] = torch.zeros(max(nq, 1), dtype=torch.float32)
        res["acc1"] = torch.zeros(nrows, 2 * I, dtype=torch.int32)
        res["h"] = torch.zeros(nrows, I, dtype=torch.float32)
        res["x2"] = torch.zeros(nrows, I, dtype=torch.int8)
        res["s2"] = torch.zeros(nrows, dtype=torch.float32)
        res["acc2"] = torch.zeros(nrows, h, dtype=torch.int32)
        res["y2"] = torch.zeros(nrows, h, dtype=torch.int16)
        for name in ("offsets", "row_of", "tk_of_row", "x_q", "x_scale", "acc1", "x2", "s2", "acc2", "y2"):
            setattr(o, name, _ptr(res[name]))
        o.h_act = _ptr(res["h"])
        if shared:
            res["xs_q"] = torch.zeros(bs, h, dtype=torch.int8)
            res["xs_scale"] = torch.zeros(bs, dtype=torch.float32)
            res["share_acc1"] = torch.zeros(bs, 2 * I, dtype=torch.int32)
            res["share_h"] = torch.zeros(bs, I, dtype=torch.float32)
            res["share_x2"] = torch.zeros(bs, I, dtype=torch.int8)
            res["share_s2"] = torch.zeros(bs, dtype=torch.float32)
            res["share_acc2"] = torch.zeros(bs, h, dtype=torch.int32)
            for name in ("xs_q", "xs_scale", "share_acc1", "share_h", "share_x2", "share_s2", "share_acc2"):
                setattr(o, name, _ptr(res[name]))
    rc = lib().oracle_forward(ctypes.byref(a), ctypes.byref(o))
    if rc:
        raise RuntimeError("oracle_forward failed: %d" % rc)
    del keep
    R = o.R
    res["R"] = R
    res["skipped"] = o.skipped
    res["output"] = _act(res["output"], fp16)
    if shared:
        res["share_output"] = _act(res["share_output"], fp16)
    if intermediates:
        res["tk_of_row"] = res["tk_of_row"][:R]
        for name in ("acc1", "h", "x2", "s2", "acc2"):
            res[name] = res[name][:R]
        if per_expert:
            res["x_q"] = res["x_q"][:R]
            res["x_scale"] = res["x_scale"][:R]
        res["y2"] = _act(res["y2"][:R], fp16)
    return res
