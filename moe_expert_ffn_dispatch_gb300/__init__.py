"""GB300 fused MoE expert block: a thin Python binding of the C ABI in
include/moe_fused.h.

Every step of the block (dispatch, quant, GEMM1 + SwiGLU, requant, GEMM2,
combine, shared expert) runs in the library's CUDA kernels.  This module only
marshals arguments: it checks tensor dtypes, shapes, devices and contiguity
and passes raw pointers.  There is no CPU path; if the shared library is
missing, loading it raises.

The functions named like the C entry points take plain integers (pointers,
sizes) and return the C status code; `MoeFused` wraps them for torch tensors.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_moe_fused.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_WORKSPACE_TOO_SMALL = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_TIMEOUT = -5
MOE_ERR_UNIMPLEMENTED = -6
MOE_ERR_ALIGNMENT = -7

# config flag: every expert on the tensor-core path with separate requant and
# combine kernels (the unfused A/B baseline); results are the same
FLAG_UNFUSED = 1
# config flag: routing weight folded into each row's GEMM2 dequant scale, the
# combine a plain sum (rounds differently from the default)
FLAG_FOLD_ROUTING = 2
# config flags, signature variants: x / output / share_output fp16; routed
# weight scales bf16 or fp16 (widened exactly); expert smooth scales [E, h]
FLAG_FP16_ACT = 4
FLAG_SCALE_BF16 = 8
FLAG_SCALE_FP16 = 16
FLAG_EXPERT_SMOOTH = 32
_SCALE_FLAGS = {torch.float32: 0, torch.bfloat16: FLAG_SCALE_BF16, torch.float16: FLAG_SCALE_FP16}

KERNEL_NAMES = ["dispatch_quant", "dispatch_finish", "expand", "gemm1_small", "gemm1_big", "requant_big",
                "gemm2_small", "gemm2_big", "combine"]
KERNEL_ID = {n: i for i, n in enumerate(KERNEL_NAMES)}
REGIONS = {"status": 0, "counts": 1, "offsets": 2, "row_of": 3, "tk_of_row": 4, "active": 5, "x_q": 6,
           "x_scale": 7, "xs_q": 8, "xs_scale": 9, "h": 10, "x2": 11, "s2": 12, "y2": 13, "slots": 14,
           "row_token": 15, "shared_row": 16, "blk_ticket": 17, "tok_ticket": 18, "tok_expect": 19,
           "ranges": 20, "x1h": 21, "x2h": 22, "dcnt": 23, "amax2": 24, "bar_tags": 25}

EXPORTS = ["moe_fused_create", "moe_fused_workspace_size", "moe_fused_forward", "moe_fused_get_status",
           "moe_fused_destroy", "moe_fused_strerror", "moe_fused_set_timing", "moe_fused_get_timing",
           "moe_fused_kernel_name", "moe_fused_dispatch_noalloc", "moe_fused_debug_region",
           "moe_fused_debug_forward_until", "moe_fused_debug_forward_range", "moe_fused_debug_gemm_acc",
           "moe_fused_debug_wait_timeout"]
DEBUG_WAIT_SITE = 240  # MOE_DEBUG_WAIT_SITE

P = ctypes.c_void_p
I32 = ctypes.c_int32


class Config(ctypes.Structure):
    _fields_ = [("bs_max", I32), ("hidden", I32), ("num_experts", I32), ("topk", I32), ("inter", I32),
                ("has_shared", I32), ("flags", I32)]


class Args(ctypes.Structure):
    _fields_ = [("x", P), ("expert_ids", P), ("expert_scales", P),
                ("gmm1_weight", P), ("gmm1_weight_scale", P), ("gmm2_weight", P), ("gmm2_weight_scale", P),
                ("share_gmm1_weight", P), ("share_gmm1_weight_scale", P),
                ("share_gmm2_weight", P), ("share_gmm2_weight_scale", P),
                ("expert_smooth_scales", P), ("share_smooth_scales", P), ("x_active_mask", P),
                ("output", P), ("share_output", P), ("expert_token_nums", P), ("bs", I32)]


class Status(ctypes.Structure):
    _fields_ = [("skipped_pairs", I32), ("error_flags", I32), ("error_site", I32),
                ("dispatched_rows", I32), ("shared_rows", I32), ("active_slots", I32),
                ("reserved", I32 * 2)]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__("%s failed: %s (%d)" % (where, strerror(code), code))
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load the CUDA library (built in-tree by __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("moe_fused CUDA library not built: %s (run __graft_entry__.build())" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name in EXPORTS:
            getattr(L, name)  # raises AttributeError if a symbol is missing
        L.moe_fused_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t)]
        L.moe_fused_workspace_size.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_size_t)]
        L.moe_fused_forward.argtypes = [P, ctypes.POINTER(Args), P, ctypes.c_size_t, P]
        L.moe_fused_get_status.argtypes = [P, P, P, ctypes.POINTER(Status)]
        L.moe_fused_destroy.argtypes = [P]
        L.moe_fused_strerror.argtypes = [ctypes.c_int]
        L.moe_fused_strerror.restype = ctypes.c_char_p
        L.moe_fused_set_timing.argtypes = [P, ctypes.c_int]
        L.moe_fused_get_timing.argtypes = [P, P, P, ctypes.c_int]
        L.moe_fused_kernel_name.argtypes = [ctypes.c_int]
        L.moe_fused_kernel_name.restype = ctypes.c_char_p
        L.moe_fused_debug_region.argtypes = [P, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t),
                                             ctypes.POINTER(ctypes.c_size_t)]
        L.moe_fused_debug_gemm_acc.argtypes = [P, ctypes.POINTER(Args), P, ctypes.c_size_t, ctypes.c_int, P, P]
        L.moe_fused_debug_wait_timeout.argtypes = [P, P, ctypes.c_size_t, ctypes.c_int, P]
        L.moe_fused_debug_forward_until.argtypes = [P, ctypes.POINTER(Args), P, ctypes.c_size_t, ctypes.c_int, P]
        L.moe_fused_debug_forward_range.argtypes = [P, ctypes.POINTER(Args), P, ctypes.c_size_t, ctypes.c_int,
                                                    ctypes.c_int, P]
        L.moe_fused_dispatch_noalloc.argtypes = [P, P, I32, I32, I32, P, P, P]
        for name in EXPORTS:
            if name not in ("moe_fused_strerror", "moe_fused_kernel_name"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


# ------------------------------------------------------------ C-named calls
def moe_fused_create(cfg: Config) -> Tuple[int, int, int]:
    h = P()
    ws = ctypes.c_size_t(0)
    rc = lib().moe_fused_create(ctypes.byref(cfg), ctypes.byref(h), ctypes.byref(ws))
    return rc, (h.value or 0), ws.value


def moe_fused_workspace_size(cfg: Config) -> Tuple[int, int]:
    ws = ctypes.c_size_t(0)
    rc = lib().moe_fused_workspace_size(ctypes.byref(cfg), ctypes.byref(ws))
    return rc, ws.value


def moe_fused_forward(handle: int, args: Args, workspace: int, workspace_bytes: int, stream: int) -> int:
    return lib().moe_fused_forward(handle, ctypes.byref(args), workspace, workspace_bytes, stream)


def moe_fused_get_status(handle: int, workspace: int, stream: int) -> Tuple[int, Status]:
    st = Status()
    rc = lib().moe_fused_get_status(handle, workspace, stream, ctypes.byref(st))
    return rc, st


def moe_fused_destroy(handle: int) -> int:
    return lib().moe_fused_destroy(handle)


def moe_fused_strerror(code: int) -> str:
    return lib().moe_fused_strerror(code).decode()


strerror = moe_fused_strerror


def moe_fused_set_timing(handle: int, enable: bool) -> int:
    return lib().moe_fused_set_timing(handle, int(enable))


def moe_fused_get_timing(handle: int, max_kernels: int = 9):
    ms = (ctypes.c_float * max_kernels)()
    n = (I32 * max_kernels)()
    rc = lib().moe_fused_get_timing(handle, ctypes.addressof(ms), ctypes.addressof(n), max_kernels)
    return rc, list(ms), list(n)


def moe_fused_kernel_name(k: int) -> str:
    return lib().moe_fused_kernel_name(k).decode()


def moe_fused_dispatch_noalloc(expert_ids: int, x_active_mask: int, bs: int, topk: int, num_experts: int,
                               expert_token_nums: int, expand_row: int, stream: int) -> int:
    """Dispatch only, with library-owned static scratch (no workspace; see the header)."""
    return lib().moe_fused_dispatch_noalloc(expert_ids, x_active_mask, bs, topk, num_experts,
                                            expert_token_nums, expand_row, stream)


def moe_fused_debug_region(handle: int, region: int) -> Tuple[int, int, int]:
    off = ctypes.c_size_t(0)
    nb = ctypes.c_size_t(0)
    rc = lib().moe_fused_debug_region(handle, region, ctypes.byref(off), ctypes.byref(nb))
    return rc, off.value, nb.value


def moe_fused_debug_forward_until(handle: int, args: Args, workspace: int, workspace_bytes: int, last_kernel: int,
                                  stream: int) -> int:
    return lib().moe_fused_debug_forward_until(handle, ctypes.byref(args), workspace, workspace_bytes, last_kernel,
                                               stream)


def moe_fused_debug_forward_range(handle: int, args: Args, workspace: int, workspace_bytes: int, first_kernel: int,
                                  last_kernel: int, stream: int) -> int:
    return lib().moe_fused_debug_forward_range(handle, ctypes.byref(args), workspace, workspace_bytes, first_kernel,
                                               last_kernel, stream)


def moe_fused_debug_gemm_acc(handle: int, args: Args, workspace: int, workspace_bytes: int, which: int,
                             acc: int, stream: int) -> int:
    return lib().moe_fused_debug_gemm_acc(handle, ctypes.byref(args), workspace, workspace_bytes, which, acc, stream)


def moe_fused_debug_wait_timeout(handle: int, workspace: int, workspace_bytes: int, which: int, stream: int) -> int:
    """Test-only: a bounded wait that runs out (0: mbarrier, 1: cross-CTA flag)."""
    return lib().moe_fused_debug_wait_timeout(handle, workspace, workspace_bytes, which, stream)


# ------------------------------------------------------------ torch wrapper
def _check(t: Optional[torch.Tensor], name: str, dtype, shape, device, optional=False) -> int:
    if t is None:
        if optional:
            return 0
        raise ValueError("%s is required" % name)
    if t.dtype != dtype:
        raise TypeError("%s: dtype %s, expected %s" % (name, t.dtype, dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s: shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.device != device:
        raise ValueError("%s: on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


class MoeFused:
    """One configured block on one CUDA device.

    Weights are passed to every forward (they stay wherever the caller keeps
    them; the library never copies them).  The workspace is a torch uint8
    tensor of `workspace_bytes`, allocated here unless the caller supplies one.
    """

    def __init__(self, bs_max: int, hidden: int, num_experts: int, topk: int, inter: int,
                 has_shared: bool, device=None, unfused: bool = False, fold_routing: bool = False,
                 act_dtype=torch.bfloat16, scale_dtype=torch.float32, expert_smooth: bool = False):
        """act_dtype: dtype of x and of the outputs (bf16 or fp16); scale_dtype:
        dtype of the routed experts' weight scales (fp32, bf16 or fp16);
        expert_smooth: expert_smooth_scales are [num_experts, hidden]."""
        self.device = torch.device(device if device is not None else "cuda")
        if self.device.type != "cuda":
            raise ValueError("the fused MoE block runs on a CUDA device only")
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        if act_dtype not in (torch.bfloat16, torch.float16):
            raise TypeError("act_dtype must be bfloat16 or float16")
        if scale_dtype not in _SCALE_FLAGS:
            raise TypeError("scale_dtype must be float32, bfloat16 or float16")
        self.act_dtype, self.scale_dtype, self.expert_smooth = act_dtype, scale_dtype, bool(expert_smooth)
        flags = ((FLAG_UNFUSED if unfused else 0) | (FLAG_FOLD_ROUTING if fold_routing else 0) |
                 (FLAG_FP16_ACT if act_dtype == torch.float16 else 0) | _SCALE_FLAGS[scale_dtype] |
                 (FLAG_EXPERT_SMOOTH if expert_smooth else 0))
        self.cfg = Config(bs_max, hidden, num_experts, topk, inter, int(bool(has_shared)), flags)
        with torch.cuda.device(self.device):
            rc, self.handle, self.workspace_bytes = moe_fused_create(self.cfg)
        if rc:
            raise MoeError(rc, "moe_fused_create")
        self._ws = None

    def __del__(self):
        h = getattr(self, "handle", 0)
        if h and _lib is not None:
            _lib.moe_fused_destroy(h)
            self.handle = 0

    # -------------------------------------------------------------- helpers
    def workspace(self) -> torch.Tensor:
        if self._ws is None:
            self._ws = torch.empty(self.workspace_bytes + 256, dtype=torch.uint8, device=self.device)
        return self._aligned(self._ws)

    @staticmethod
    def _aligned(buf: torch.Tensor) -> torch.Tensor:
        off = (-buf.data_ptr()) % 256
        return buf[off:]

    def make_args(self, x, expert_ids, expert_scales, w1, w1_scale, w2, w2_scale,
                  share_w1=None, share_w1_scale=None, share_w2=None, share_w2_scale=None,
                  smooth=None, share_smooth=None, mask=None, out=None, share_out=None, token_nums=None):
        c, dev = self.cfg, self.device
        bs = x.shape[0]
        h, E, K, I = c.hidden, c.num_experts, c.topk, c.inter
        act, sdt = self.act_dtype, self.scale_dtype
        if out is None:
            out = torch.empty(bs, h, dtype=act, device=dev)
        if share_out is None and c.has_shared:
            share_out = torch.empty(bs, h, dtype=act, device=dev)
        if token_nums is None:
            token_nums = torch.empty(E, dtype=torch.int32, device=dev)
        a = Args()
        a.x = _check(x, "x", act, (bs, h), dev)
        a.expert_ids = _check(expert_ids, "expert_ids", torch.int32, (bs, K), dev)
        a.expert_scales = _check(expert_scales, "expert_scales", torch.float32, (bs, K), dev)
        a.gmm1_weight = _check(w1, "gmm1_weight", torch.int8, (E, 2 * I, h), dev)
        a.gmm1_weight_scale = _check(w1_scale, "gmm1_weight_scale", sdt, (E, 2 * I), dev)
        a.gmm2_weight = _check(w2, "gmm2_weight", torch.int8, (E, h, I), dev)
        a.gmm2_weight_scale = _check(w2_scale, "gmm2_weight_scale", sdt, (E, h), dev)
        opt = not c.has_shared
        a.share_gmm1_weight = _check(share_w1, "share_gmm1_weight", torch.int8, (2 * I, h), dev, opt)
        a.share_gmm1_weight_scale = _check(share_w1_scale, "share_gmm1_weight_scale", torch.float32, (2 * I,), dev, opt)
        a.share_gmm2_weight = _check(share_w2, "share_gmm2_weight", torch.int8, (h, I), dev, opt)
        a.share_gmm2_weight_scale = _check(share_w2_scale, "share_gmm2_weight_scale", torch.float32, (h,), dev, opt)
        a.expert_smooth_scales = _check(smooth, "expert_smooth_scales", torch.float32,
                                        (E, h) if self.expert_smooth else (h,), dev, True)
        a.share_smooth_scales = _check(share_smooth, "share_smooth_scales", torch.float32, (h,), dev, True)
        if mask is not None and mask.dtype == torch.bool:
            mask = mask.view(torch.uint8)
        a.x_active_mask = _check(mask, "x_active_mask", torch.uint8, (bs,), dev, True)
        a.output = _check(out, "output", act, (bs, h), dev)
        a.share_output = _check(share_out, "share_output", act, (bs, h), dev, True)
        a.expert_token_nums = _check(token_nums, "expert_token_nums", torch.int32, (E,), dev)
        a.bs = bs
        keep = (x, expert_ids, expert_scales, w1, w1_scale, w2, w2_scale, share_w1, share_w1_scale, share_w2,
                share_w2_scale, smooth, share_smooth, mask, out, share_out, token_nums)
        return a, keep, (out, share_out, token_nums)

    def forward(self, x, expert_ids, expert_scales, w1, w1_scale, w2, w2_scale, share_w1=None,
                share_w1_scale=None, share_w2=None, share_w2_scale=None, smooth=None, share_smooth=None,
                mask=None, out=None, share_out=None, token_nums=None, workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None, until: Optional[int] = None,
                start: Optional[int] = None):
        """Enqueue one forward; returns (output, share_output or None, expert_token_nums).
        `until` (test use) stops after that kernel id, `start` (test use) starts
        at that kernel id on the state the workspace holds
        (moe_fused_debug_forward_range)."""
        a, keep, outs = self.make_args(x, expert_ids, expert_scales, w1, w1_scale, w2, w2_scale, share_w1,
                                       share_w1_scale, share_w2, share_w2_scale, smooth, share_smooth, mask,
                                       out, share_out, token_nums)
        ws = self.workspace() if workspace is None else workspace
        s = (stream if stream is not None else torch.cuda.current_stream(self.device)).cuda_stream
        if until is None and start is None:
            rc = moe_fused_forward(self.handle, a, ws.data_ptr(), ws.numel(), s)
        else:
            first = 0 if start is None else start
            last = len(KERNEL_NAMES) - 1 if until is None else until
            rc = moe_fused_debug_forward_range(self.handle, a, ws.data_ptr(), ws.numel(), first, last, s)
        if rc:
            raise MoeError(rc, "moe_fused_forward")
        del keep
        return outs

    def forward_inputs(self, inp, weights, **kw):
        """Forward on a synthetic input bundle (device tensors) and a weights dict."""
        return self.forward(inp["x"], inp["expert_ids"], inp["expert_scales"], weights["w1"], weights["w1_scale"],
                            weights["w2"], weights["w2_scale"], weights.get("share_w1"),
                            weights.get("share_w1_scale"), weights.get("share_w2"), weights.get("share_w2_scale"),
                            weights.get("smooth"), weights.get("share_smooth"), inp.get("mask"), **kw)

    def status(self, workspace: Optional[torch.Tensor] = None, stream=None) -> Dict[str, int]:
        ws = self.workspace() if workspace is None else workspace
        s = (stream if stream is not None else torch.cuda.current_stream(self.device)).cuda_stream
        rc, st = moe_fused_get_status(self.handle, ws.data_ptr(), s)
        d = {"rc": rc, "skipped_pairs": st.skipped_pairs, "error_flags": st.error_flags,
             "error_site": st.error_site, "dispatched_rows": st.dispatched_rows,
             "shared_rows": st.shared_rows, "active_slots": st.active_slots}
        return d

    def set_timing(self, enable: bool):
        rc = moe_fused_set_timing(self.handle, enable)
        if rc:
            raise MoeError(rc, "moe_fused_set_timing")

    def get_timing(self) -> Dict[str, Tuple[float, int]]:
        rc, ms, n = moe_fused_get_timing(self.handle, len(KERNEL_NAMES))
        if rc < 0:
            raise MoeError(rc, "moe_fused_get_timing")
        return {KERNEL_NAMES[k]: (ms[k], n[k]) for k in range(len(KERNEL_NAMES))}

    def region(self, name: str, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
        """A uint8 view of one workspace region (test use)."""
        rc, off, nb = moe_fused_debug_region(self.handle, REGIONS[name])
        if rc:
            raise MoeError(rc, "moe_fused_debug_region")
        ws = self.workspace() if workspace is None else workspace
        return ws[off:off + nb]

    def debug_gemm_acc(self, which: int, acc: torch.Tensor, *fargs, workspace=None, **fkw):
        a, keep, _ = self.make_args(*fargs, **fkw)
        ws = self.workspace() if workspace is None else workspace
        s = torch.cuda.current_stream(self.device).cuda_stream
        if acc.dtype != torch.int32 or acc.device != self.device or not acc.is_contiguous():
            raise ValueError("acc must be a contiguous int32 tensor on the block's device")
        rc = moe_fused_debug_gemm_acc(self.handle, a, ws.data_ptr(), ws.numel(), which, acc.data_ptr(), s)
        if rc:
            raise MoeError(rc, "moe_fused_debug_gemm_acc")
        del keep


def _packed(specs, device, pinned: bool = False):
    """Tensors of `specs` [(name, shape, dtype)] as views into one buffer,
    each starting on a 256-byte boundary: one copy moves them all."""
    offs, off = [], 0
    for name, shape, dtype in specs:
        n = int(torch.Size(shape).numel()) * torch.empty(0, dtype=dtype).element_size()
        offs.append((name, shape, dtype, off, n))
        off += (n + 255) // 256 * 256
    buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = {name: buf[o:o + n].view(dtype).view(shape) for name, shape, dtype, o, n in offs}
    return buf, views


class GraphedStep:
    """One whole inference step captured as a CUDA graph: one host-to-device
    copy of this step's inputs (packed in one pinned buffer), the forward, and
    one device-to-host copy of output, share_output and expert_token_nums
    (packed likewise).  For serving loops with a fixed batch shape: write the
    next step's inputs into `host_inputs` in place, call `run()`, synchronise
    `stream`, read `host_outputs`.

    host_inputs: dict with "x", "expert_ids", "expert_scales" and optionally
    "mask" (CPU tensors of the block's dtypes and shapes, bs <= bs_max); their
    values are copied into the step's own pinned buffer, whose views become
    `self.host_inputs`.  weights: dict as for MoeFused.forward_inputs (device
    tensors, not copied).
    """

    def __init__(self, blk: MoeFused, host_inputs: Dict[str, torch.Tensor], weights: Dict[str, torch.Tensor],
                 stream: Optional[torch.cuda.Stream] = None):
        self.blk = blk
        self.weights = weights
        dev = blk.device
        specs = [(k, tuple(v.shape), v.dtype) for k, v in host_inputs.items()]
        self._hin, self.host_inputs = _packed(specs, "cpu", pinned=True)
        self._din, self.dev_inputs = _packed(specs, dev)
        for k, v in host_inputs.items():
            self.host_inputs[k].copy_(v)
        bs, h = host_inputs["x"].shape
        ospecs = [("output", (bs, h), blk.act_dtype), ("expert_token_nums", (blk.cfg.num_experts,), torch.int32)]
        if blk.cfg.has_shared:
            ospecs.append(("share_output", (bs, h), blk.act_dtype))
        self._dout, self.dev_outputs = _packed(ospecs, dev)
        self._hout, self.host_outputs = _packed(ospecs, "cpu", pinned=True)
        self.stream = stream if stream is not None else torch.cuda.Stream(device=dev)
        blk.workspace()  # allocated before the capture
        with torch.cuda.stream(self.stream):
            self._step()  # eager once: builds the tensor maps, checks the arguments
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._step()
        self.stream.synchronize()

    def _step(self):
        self._din.copy_(self._hin, non_blocking=True)
        o = self.dev_outputs
        self.blk.forward_inputs(self.dev_inputs, self.weights, out=o["output"], share_out=o.get("share_output"),
                                token_nums=o["expert_token_nums"])
        self._hout.copy_(self._dout, non_blocking=True)

    def run(self):
        """Replay the step, asynchronous on `self.stream` (synchronise that
        stream before reading host_outputs)."""
        with torch.cuda.stream(self.stream):
            self.graph.replay()

    def h2d_bytes(self) -> int:
        """Bytes of this step's inputs (the packed copy moves these plus alignment padding)."""
        return sum(v.numel() * v.element_size() for v in self.host_inputs.values())

    def d2h_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.host_outputs.values())


class PipelinedStep:
    """A serving loop whose host copies overlap the neighbouring steps'
    forwards.  Step k uses buffer set k % depth (each set: pinned host inputs
    and outputs, packed device inputs and outputs, and a CUDA graph of the
    forward on them).  submit() enqueues, for the step's set:
      * the packed host-to-device copy of its inputs, on the copy-in stream,
        once the forward that last read that set's device inputs is done;
      * its forward (the set's graph), on the compute stream, once those
        inputs have landed and the copy that last read the set's device
        outputs is done -- forwards run one after another on this stream,
        sharing the block's workspace;
      * the packed device-to-host copy of its outputs, on the copy-out
        stream, once the forward is done.
    So while step k computes, step k + 1's inputs and step k - 1's outputs
    move.  Every step still copies all of its inputs in and all of its outputs
    out.

    host_inputs: initial values of every set's inputs (as for GraphedStep).
    Before writing step k's inputs, take the views from inputs_for(k) (it
    waits until that set's previous input copy has left the buffer).
    result(k) waits for step k's outputs and returns the set's host output
    views, valid until step k + depth is submitted.
    """

    def __init__(self, blk: MoeFused, host_inputs: Dict[str, torch.Tensor], weights: Dict[str, torch.Tensor],
                 depth: int = 2):
        if depth < 2:
            raise ValueError("depth must be at least 2")
        self.blk, self.weights, self.depth = blk, weights, depth
        dev = blk.device
        specs = [(k, tuple(v.shape), v.dtype) for k, v in host_inputs.items()]
        bs, h = host_inputs["x"].shape
        ospecs = [("output", (bs, h), blk.act_dtype), ("expert_token_nums", (blk.cfg.num_experts,), torch.int32)]
        if blk.cfg.has_shared:
            ospecs.append(("share_output", (bs, h), blk.act_dtype))
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_comp = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        blk.workspace()  # allocated before the captures
        self.sets = []
        for _ in range(depth):
            st = {}
            st["hin_buf"], st["hin"] = _packed(specs, "cpu", pinned=True)
            st["din_buf"], st["din"] = _packed(specs, dev)
            st["dout_buf"], st["dout"] = _packed(ospecs, dev)
            st["hout_buf"], st["hout"] = _packed(ospecs, "cpu", pinned=True)
            for k, v in host_inputs.items():
                st["hin"][k].copy_(v)
            st["din_buf"].copy_(st["hin_buf"])
            for name in ("ev_in", "ev_fwd", "ev_out"):
                st[name] = torch.cuda.Event()
            with torch.cuda.stream(self.s_comp):
                self._forward(st)  # eager once: builds the tensor maps, checks the arguments
            self.s_comp.synchronize()
            st["graph"] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(st["graph"], stream=self.s_comp):
                self._forward(st)
            self.s_comp.synchronize()
            self.sets.append(st)
        self.submitted = 0

    def _forward(self, st):
        o = st["dout"]
        self.blk.forward_inputs(st["din"], self.weights, out=o["output"], share_out=o.get("share_output"),
                                token_nums=o["expert_token_nums"])

    def inputs_for(self, k: int) -> Dict[str, torch.Tensor]:
        """Host input views of step k's set, once its previous copy-in is done."""
        st = self.sets[k % self.depth]
        st["ev_in"].synchronize()
        return st["hin"]

    def submit(self) -> int:
        """Enqueue the next step; returns its index."""
        k = self.submitted
        st = self.sets[k % self.depth]
        self.s_in.wait_event(st["ev_fwd"])    # the set's device inputs are free
        with torch.cuda.stream(self.s_in):
            st["din_buf"].copy_(st["hin_buf"], non_blocking=True)
            st["ev_in"].record(self.s_in)
        self.s_comp.wait_event(st["ev_in"])
        self.s_comp.wait_event(st["ev_out"])  # the set's device outputs are free
        with torch.cuda.stream(self.s_comp):
            st["graph"].replay()
            st["ev_fwd"].record(self.s_comp)
        self.s_out.wait_event(st["ev_fwd"])
        with torch.cuda.stream(self.s_out):
            st["hout_buf"].copy_(st["dout_buf"], non_blocking=True)
            st["ev_out"].record(self.s_out)
        self.submitted = k + 1
        return k

    def result(self, k: int) -> Dict[str, torch.Tensor]:
        """Host output views of step k (waits for its copy-out)."""
        if not (self.submitted - self.depth <= k < self.submitted):
            raise ValueError("step %d is not among the last %d submitted" % (k, self.depth))
        st = self.sets[k % self.depth]
        st["ev_out"].synchronize()
        return st["hout"]

    def h2d_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.sets[0]["hin"].values())

    def d2h_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.sets[0]["hout"].values())
