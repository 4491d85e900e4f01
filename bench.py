"""Benchmark of the fused MoE expert block on GB300.

One step = one forward of the whole block (dispatch, quant, GEMM1 + SwiGLU,
requant, GEMM2, combine, shared expert) on one batch, with weights and inputs
already resident in HBM.  The default batch is the largest single-GPU
workload, prefill: bs 4096 tokens, h 4096, 256 experts, top-8 with balanced
routing (128 rows per expert), I 2048, shared expert.  `--workload` selects
the others (tiny, decode8, decode64, mid512).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (torchrun): each rank runs an independent replica on its own batch
(no collective on the data path; weak scaling); the timed region is bracketed
by a barrier and the max over ranks is reported.

`--impl reference` times the CPU oracle on the host cores on a bounded sample
of the same workload (the only other reference available for this block).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE block tokens/s and µs/forward at 1 GB300; % of HBM / INT8 roofline"
PROFILES = os.path.join(ROOT, "profiles")


# ---------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _code_only(src: str) -> str:
    """C / CUDA source without comments and with whitespace collapsed (string
    and character literals, e.g. inline PTX, kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sha(kernel: str) -> str:
    """Hash of the code (comments and layout ignored) of the kernel's source
    file and the headers it includes: ncu counters taken on one version stay
    valid for another that differs only in comments."""
    csrc = os.path.join(ROOT, "moe_expert_ffn_dispatch_gb300", "csrc")
    hsh = hashlib.sha256()
    for name in (KERNEL_SOURCES[kernel], "device_prims.cuh", "epilogue_ops.cuh", "moe_internal.h", "quant_ops.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            hsh.update(_code_only(f.read()).encode())
    return hsh.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    profiles/<kernel>_<workload>.md, if it was taken on the current kernel
    source (matching kernel_sha); else None."""
    path = os.path.join(PROFILES, "%s_%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m1 = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    m2 = re.search(r"kernel_sha:\s*([0-9a-f]+)", txt)
    if not m1 or not m2 or m2.group(1) != kernel_sha(kernel):
        return None
    return int(m1.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []
        self._reader = None

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line)

    def __enter__(self):
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()
        # the timed region starts only once the sampler has started sampling
        # (its driver initialisation then no longer overlaps the timed launches)
        t0 = time.monotonic()
        while not self.lines and self.proc.poll() is None and time.monotonic() - t0 < 5.0:
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self._reader is not None:
                self._reader.join(timeout=5)
        return False

    def summary(self):
        sm, smax, reasons = [], [], 0
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                reasons |= int(parts[3], 16)
            except (ValueError, IndexError):
                continue
        names = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
                 0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
        rs = [n for b, n in names.items() if reasons & b]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": rs, "samples": len(sm)}


SMALL_ROWS = 8  # experts with at most this many rows run in the weight-streaming kernels


def algorithmic_bytes(wl, counts_per_expert, n_active, unfused=False):
    """Bytes (and int ops) each kernel must handle at least once: the roofline numerator.

    Per touched expert (routed experts with >= 1 row, plus the shared expert
    when it has rows) GEMM1 reads W1 (2I*h int8) and its scales (2I fp32) and
    GEMM2 reads W2 (h*I int8) and its scales (h fp32).  Activations count at
    the sizes the method defines, once per kernel that consumes or produces
    them; scratch round trips (the fp32 h read back by a fused requant, y2 read
    back by a fused combine, f16 operand copies) are not algorithmic.
      gemm1_small  W1 + m*(h x_q in + I x2 out + 4 s2 out)      (requant fused)
      gemm1_big    W1 + m*(h x_q in + 4I h out)
      requant_big  m*(4I h in + I x2 out + 4 s2 out)
      gemm2_small  W2 + m*(I + 4 in) + 2h per shared row, + 2h*bs out when it combines
      gemm2_big    W2 + m*(I + 4 in + 2h y2 out)
      combine      2h per routed row in + 2h*bs out
    Experts with at most SMALL_ROWS rows (when h, I <= 4096 and the forward
    is not the unfused A/B chain) run in the *_small kernels, the others in
    the tensor-core *_big kernels.  The step
    total counts weights once plus the block's own inputs and outputs."""
    h, I, K, bs = wl.hidden, wl.inter, wl.topk, wl.bs
    small_ok = h <= 4096 and I <= 4096 and not unfused
    groups = [(c, True) for c in counts_per_expert if c > 0]
    shared = n_active if (wl.has_shared and n_active > 0) else 0
    if shared:
        groups.append((shared, False))
    keys = ["gemm1_small", "gemm1_big", "gemm2_small", "gemm2_big", "requant_big", "combine"]
    out = {k: 0 for k in keys}
    ops = {k: 0 for k in keys}
    any_big = False
    for m, routed in groups:
        # a batch of at most SMALL_ROWS tokens runs every expert in the *_small
        # kernels (more rows, from repeated ids, in several slots; the weights
        # still count once here)
        small = small_ok and (m <= SMALL_ROWS or bs <= SMALL_ROWS)
        any_big |= not small
        if small:
            out["gemm1_small"] += 2 * I * h + 8 * I + m * (h + I + 4)
            out["gemm2_small"] += h * I + 4 * h + m * (I + 4) + (0 if routed else m * 2 * h)
        else:
            out["gemm1_big"] += 2 * I * h + 8 * I + m * (h + 4 * I)
            out["requant_big"] += m * (4 * I + I + 4)
            out["gemm2_big"] += h * I + 4 * h + m * (I + 4 + 2 * h)
        g = "small" if small else "big"
        ops["gemm1_" + g] += 2 * m * 2 * I * h
        ops["gemm2_" + g] += 2 * m * h * I
    routed_rows = sum(m for m, r in groups if r)
    if any_big:
        out["combine"] += routed_rows * 2 * h + bs * 2 * h
    else:
        out["gemm2_small"] += bs * 2 * h  # the small GEMM2 combines every token
    touched = len(groups)
    rows = sum(m for m, _ in groups)
    out["step"] = touched * (2 * I * h + h * I + 4 * (2 * I + h)) + bs * h * 2 + bs * K * 8 + \
        bs * h * 2 * (2 if wl.has_shared else 1) + wl.num_experts * 4
    out["int_ops"] = 2 * rows * (2 * I * h + h * I)
    out["ops"] = ops
    out["touched_experts"] = touched
    out["rows"] = rows
    return out


def roofline_of(bytes_, ops, seconds, peaks):
    """Bound = the larger of T_mem (bytes at the measured HBM copy rate) and
    T_ops (int ops at the measured dense bf16 rate: the exact int8 products run
    as f16 codes on the tensor cores, whose f16 rate equals the bf16 rate)."""
    t_mem = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_ops = ops / (peaks["bf16_tflops"] * 1e12)
    if t_ops > t_mem:
        return {"bound": "tensor", "achieved": ops / seconds / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": t_ops / seconds}
    return {"bound": "hbm", "achieved": bytes_ / seconds / 1e9, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": t_mem / seconds}


KERNEL_SOURCES = {"gemm1_small": "moe_gemm.cu", "gemm2_small": "moe_gemm.cu",
                  "gemm1_big": "tc_gemm.cu", "gemm2_big": "tc_gemm.cu"}


# ---------------------------------------------------------------- our arm
# ---------------------------------------------------------------- replicas
def rank_workload(wl, rank):
    """The batch rank `rank` runs: same shapes and weights, its own token draw
    (the path shards by independent batches; there is no data-path collective)."""
    return synth.Workload(**{**wl.__dict__, "seed": wl.seed + 7919 * rank})


def max_over_ranks(x, device="cpu"):
    """The slowest rank's value (the job ends when the last replica does)."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def workload_config(wl, alg, ws):
    return {"workload": wl.name, "bs": wl.bs, "hidden": wl.hidden, "experts": wl.num_experts,
            "topk": wl.topk, "inter": wl.inter, "shared_expert": wl.has_shared,
            "touched_experts": alg["touched_experts"], "rows": alg["rows"],
            "l2": "inputs larger than L2 (%.2f GB of touched weights per step vs 0.13 GB L2)" % (alg["step"] / 1e9),
            "parallelism": "replicas x%d (independent batches, no collective)" % ws}


def host_alg(wl):
    """algorithmic_bytes from the seeded routing, computed on the host."""
    inp = synth.make_inputs(wl, with_weights=False)
    act = torch.ones(wl.bs, dtype=torch.bool) if inp.mask is None else inp.mask.bool()
    ids = inp.expert_ids[act].flatten()
    ids = ids[(ids >= 0) & (ids < wl.num_experts)]
    counts = torch.bincount(ids.long(), minlength=wl.num_experts).tolist()
    return algorithmic_bytes(wl, counts, int(act.sum()))


def per_forward_summary(us):
    """Median, 10th and 90th percentile (nearest rank) of per-forward times."""
    v = sorted(us)
    if not v:
        return {"median": None, "p10": None, "p90": None}

    def rank(q):
        return v[min(len(v) - 1, max(0, math.ceil(q * len(v)) - 1))]
    return {"median": statistics.median(v), "p10": rank(0.10), "p90": rank(0.90)}


def whole_job_tokens_per_s(bs, world_size, steps, seconds):
    """Tokens all ranks processed divided by the (max-over-ranks) time."""
    return bs * world_size * steps / seconds


def run_ours(args, wl, ws, rank, local):
    import moe_expert_ffn_dispatch_gb300 as m

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        torch.distributed.init_process_group("nccl")
    # each rank runs its own batch (seed + rank) through the same replicated weights
    inp = synth.make_inputs(rank_workload(wl, rank), with_weights=False)
    base = synth.make_inputs(wl, with_weights=False)
    weights = {"w1": synth.draw_all_w1(wl, dev), "w1_scale": base.w1_scale.to(dev),
               "w2": synth.draw_all_w2(wl, dev), "w2_scale": base.w2_scale.to(dev)}
    if wl.has_shared:
        weights.update(share_w1=synth.draw_w1(wl, wl.num_experts, dev), share_w1_scale=base.share_w1_scale.to(dev),
                       share_w2=synth.draw_w2(wl, wl.num_experts, dev), share_w2_scale=base.share_w2_scale.to(dev))
    if base.smooth is not None:
        weights["smooth"] = base.smooth.to(dev)
    if base.share_smooth is not None:
        weights["share_smooth"] = base.share_smooth.to(dev)
    di = {"x": inp.x.to(dev), "expert_ids": inp.expert_ids.to(dev), "expert_scales": inp.expert_scales.to(dev)}
    if inp.mask is not None:
        di["mask"] = inp.mask.to(dev)

    blk = m.MoeFused(wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter, wl.has_shared, dev,
                     unfused=getattr(args, "unfused", False), fold_routing=getattr(args, "fold_routing", False))
    stream = torch.cuda.current_stream(dev)
    out, sout, nums = blk.forward_inputs(di, weights)
    torch.cuda.synchronize()
    st = blk.status()
    if st["rc"] != 0:
        raise RuntimeError("forward status %s" % st)
    counts = nums.cpu().tolist()
    n_active = int(inp.mask.sum()) if inp.mask is not None else wl.bs
    alg = algorithmic_bytes(wl, counts, n_active, unfused=getattr(args, "unfused", False))

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    # ---- device-resident timing (value): K forwards back to back, no instrumentation
    for _ in range(args.warmup):
        blk.forward_inputs(di, weights, out=out, share_out=sout, token_nums=nums)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            blk.forward_inputs(di, weights, out=out, share_out=sout, token_nums=nums)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = e0.elapsed_time(e1)
    if blk.status()["rc"] != 0:
        raise RuntimeError("device status after the timed loop: %s" % blk.status())
    ms_total = max_over_ranks(ms_total, dev)

    # ---- per-kernel durations: a second pass of the same K forwards with CUDA
    # events around every launch on the launch stream (events between the
    # launches serialise them, so this pass does not give the headline)
    blk.set_timing(True)
    blk.get_timing()  # clear
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        blk.forward_inputs(di, weights, out=out, share_out=sout, token_nums=nums)
    e3.record(stream)
    torch.cuda.synchronize()
    ms_instrumented = e2.elapsed_time(e3)
    ktimes = blk.get_timing()
    # how the last forward split the CTAs between the two GEMM engines
    hdr = blk.region("slots")[:32].view(torch.int32).cpu().tolist()
    n_ctas = min(torch.cuda.get_device_properties(dev).multi_processor_count, 1023)
    engines = {"side_by_side": bool(hdr[6]), "small_phase_ctas": hdr[5],
               "tensor_core_ctas": (n_ctas - hdr[5]) if hdr[6] else n_ctas}
    # the small experts' GEMM2 streams behind their GEMM1 in one launch: that
    # launch carries both GEMMs' algorithmic bytes and ops
    streamed_small = ktimes["gemm1_small"][1] > 0 and ktimes["gemm2_small"][1] == 0
    # a batch of at most 8 tokens: the gemm1_small launch is the whole forward
    # (dispatch and quant included; its bytes and ops are the forward's)
    one_launch = streamed_small and ktimes["dispatch_quant"][1] == 0
    if one_launch:
        # x in, ids and routing weights in, expert_token_nums out
        alg["gemm1_small"] += wl.bs * wl.hidden * 2 + wl.bs * wl.topk * 8 + wl.num_experts * 4
    if streamed_small:
        alg["gemm1_small"] += alg["gemm2_small"]
        alg["ops"]["gemm1_small"] += alg["ops"]["gemm2_small"]
        alg["gemm2_small"] = 0
        alg["ops"]["gemm2_small"] = 0
    blk.set_timing(False)
    launches = sum(n for _, n in ktimes.values())  # the timed pass launches the same kernels

    # ---- per-forward distribution: a third pass of the same K forwards with a
    # pair of events around each forward (an event between two forwards ends
    # the overlap of one forward's last kernel with the next one's first, so
    # this pass gives the spread, not the headline)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_ev, b_ev in ev:
        a_ev.record(stream)
        blk.forward_inputs(di, weights, out=out, share_out=sout, token_nums=nums)
        b_ev.record(stream)
    torch.cuda.synchronize()
    per_fwd = per_forward_summary([a_ev.elapsed_time(b_ev) * 1e3 for a_ev, b_ev in ev])

    # ---- end to end through the public API: host inputs in, host results out.
    # The serving loop is the API's PipelinedStep: every step copies its packed
    # inputs in from pinned host memory, runs the forward (a CUDA graph per
    # buffer set) and copies its packed outputs back; with two buffer sets a
    # step's copies overlap its neighbours' forwards.  If that cannot be built,
    # the one-graph GraphedStep (copies serialised with the forward), and if
    # capture fails, eager calls.  The timed region ends when the last step's
    # outputs are in host memory.
    pin = {k: v.cpu().pin_memory() for k, v in di.items()}
    e2e_sync = None
    try:
        pstep = m.PipelinedStep(blk, pin, weights)
        h2d, d2h = pstep.h2d_bytes(), pstep.d2h_bytes()
        e2e_path = ("pipelined steps (two buffer sets; copy-in, compute and copy-out streams): per step one packed "
                    "H2D copy of the inputs, the forward as a CUDA graph, one packed D2H copy of the outputs, a "
                    "step's copies overlapping its neighbours' forwards")

        def e2e_step():
            pstep.submit()

        def e2e_sync():
            pstep.result(pstep.submitted - 1)
    except RuntimeError as err:
        pipe_err = str(err).splitlines()[0][:120]
        try:
            gstep = m.GraphedStep(blk, pin, weights)
            h2d, d2h = gstep.h2d_bytes(), gstep.d2h_bytes()
            e2e_path = ("cuda graph: one packed H2D copy of the inputs, the forward, one packed D2H copy of the "
                        "outputs (pipelined steps failed: %s)" % pipe_err)

            def e2e_step():
                gstep.run()
                gstep.stream.synchronize()
        except RuntimeError as err2:
            h_out = torch.empty_like(out, device="cpu").pin_memory()
            h_sout = torch.empty_like(sout, device="cpu").pin_memory() if sout is not None else None
            h_nums = torch.empty_like(nums, device="cpu").pin_memory()
            h2d = sum(v.numel() * v.element_size() for v in pin.values())
            d2h = h_out.numel() * 2 + (h_sout.numel() * 2 if h_sout is not None else 0) + h_nums.numel() * 4
            e2e_path = "eager calls (graph capture failed: %s)" % str(err2).splitlines()[0][:120]

            def e2e_step():
                for k, v in pin.items():
                    di[k].copy_(v, non_blocking=True)
                blk.forward_inputs(di, weights, out=out, share_out=sout, token_nums=nums)
                h_out.copy_(out, non_blocking=True)
                if h_sout is not None:
                    h_sout.copy_(sout, non_blocking=True)
                h_nums.copy_(nums, non_blocking=True)
                stream.synchronize()

    for _ in range(args.warmup):
        e2e_step()
    if e2e_sync is not None:
        e2e_sync()
    barrier()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 200))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    if e2e_sync is not None:
        e2e_sync()
    t1 = time.perf_counter()
    barrier()
    e2e_s = max_over_ranks(t1 - t0, dev)

    peaks, peak_kind = measured_peaks()
    # dominant kernel: the GEMM kernel with the most work, i.e. the largest
    # roofline time max(bytes / HBM rate, ops / tensor rate) (with the engines
    # side by side, launch durations overlap and no longer rank the kernels)
    def ideal_s(k):
        return max(alg[k] / (peaks["hbm_gbs"] * 1e9), alg["ops"][k] / (peaks["bf16_tflops"] * 1e12))

    launched = [k for k in KERNEL_SOURCES if ktimes[k][1] > 0] or list(KERNEL_SOURCES)
    dom = max(launched, key=ideal_s)
    d_ms, d_n = ktimes[dom]
    d_avg_s = d_ms / max(d_n, 1) / 1e3
    roof = roofline_of(alg[dom], alg["ops"][dom], d_avg_s, peaks)
    traffic = recorded_traffic(dom, wl.name)
    step_s = ms_total / args.steps / 1e3
    tokens = wl.bs * ws
    res = {
        "metric": METRIC,
        "value": whole_job_tokens_per_s(wl.bs, ws, args.steps, ms_total / 1e3),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_total / args.steps,
        "us_per_forward": ms_total / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": "synthetic (seeded counter-hash inputs, random-init int8 weights)",
        "config": {**workload_config(wl, alg, ws), **({"unfused": True} if getattr(args, "unfused", False) else {}),
                   **({"fold_routing": True} if getattr(args, "fold_routing", False) else {})},
        "roofline": {**roof, "traffic": traffic, "kernel": dom, "peak_kind": peak_kind,
                     "streamed_small_gemm2": streamed_small, "one_launch_forward": one_launch,
                     "alg_bytes_per_launch": alg[dom], "int_ops_per_launch": alg["ops"][dom],
                     "avg_launch_us": d_avg_s * 1e6,
                     "timing": "CUDA events around each launch, second pass of the same %d forwards "
                               "(%.1f us per forward instrumented)" % (args.steps, ms_instrumented / args.steps * 1e3)},
        "roofline_step": {**roofline_of(alg["step"], alg["int_ops"], ms_total / args.steps / 1e3, peaks),
                          "alg_bytes": alg["step"], "int_ops": alg["int_ops"]},
        "per_forward_us": {**per_fwd, "timing": "CUDA events around each forward, third pass of the same %d "
                                               "forwards" % args.steps},
        "kernels_us": {k: (v[0] / max(v[1], 1) * 1e3) for k, v in ktimes.items()},
        "engines": engines,
        "gpu_launches": launches,
        "e2e": {"value": whole_job_tokens_per_s(wl.bs, ws, e2e_steps, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "path": e2e_path},
        "clocks": clk.summary(),
    }
    if inp.mask is not None:
        # masked workloads: tokens that take part in the block (inactive ones only get zero rows)
        res["active_tokens_per_s"] = whole_job_tokens_per_s(n_active, ws, args.steps, ms_total / 1e3)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
        if args.cpu_full:
            res["cpu_baseline"]["full_forward"] = cpu_full_forward(wl)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return res if rank == 0 else None


# ---------------------------------------------------------------- oracle arms
def _oracle_setup(wl):
    import oracle
    inp = synth.make_inputs(wl, with_weights=False)
    cache = {}
    need = synth.touched_experts(inp.expert_ids, wl.num_experts, inp.mask)
    for e in need + ([wl.num_experts] if wl.has_shared else []):
        cache[e] = (synth.draw_w1(wl, e), synth.draw_w2(wl, e))
    return oracle, inp, cache


def cpu_baseline(wl, budget_s=15.0):
    """The oracle as it stands, on the host cores, on a bounded sample of about
    `budget_s` seconds: whole forwards of the workload for batches of at most
    512 tokens; for larger batches (prefill) forwards restricted to
    consecutive 32-token samples in turn (the oracle's token_sample: dispatch
    and quant of every token, the GEMMs and combine of the sampled tokens),
    counting the active sampled tokens."""
    oracle, inp, cache = _oracle_setup(wl)
    threads = os.cpu_count() or 1
    bs = wl.bs
    chunk = bs if bs <= 512 else 32
    mask = torch.ones(bs, dtype=torch.bool) if inp.mask is None else inp.mask.bool()
    n, n_tok, t0 = 0, 0, time.perf_counter()
    while True:
        if chunk == bs:
            oracle.forward(inp, threads=threads, expert_weights=lambda e: cache[e])
            n_tok += bs
        else:
            samp = torch.zeros(bs, dtype=torch.bool)
            lo = (n * chunk) % bs
            samp[lo:lo + chunk] = True
            oracle.forward(inp, threads=threads, token_sample=samp, expert_weights=lambda e: cache[e])
            n_tok += int((samp & mask).sum())
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    if chunk == bs:
        sample = "%d full forwards of %s (bs %d), weights pre-drawn on the host" % (n, wl.name, bs)
    else:
        sample = ("%d forwards of %s (bs %d) restricted to %d-token samples (%d tokens: dispatch and quant of "
                  "every token, GEMMs and combine of the sampled tokens' %d routed rows and shared row), "
                  "weights pre-drawn on the host" % (n, wl.name, bs, chunk, n_tok, wl.topk))
    return {"value": n_tok / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample}


def cpu_full_forward(wl):
    """One whole forward of the workload by the oracle on the host cores
    (every token, every row; weights drawn on the host before the clock starts)."""
    oracle, inp, cache = _oracle_setup(wl)
    threads = os.cpu_count() or 1
    n_act = wl.bs if inp.mask is None else int(inp.mask.bool().sum())
    t0 = time.perf_counter()
    oracle.forward(inp, threads=threads, intermediates=False, expert_weights=lambda e: cache[e])
    dt = time.perf_counter() - t0
    return {"seconds": dt, "value": n_act / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "one full forward of %s (bs %d): every token and row, weights pre-drawn on the host"
                      % (wl.name, wl.bs)}


def run_reference(args, wl, ws, rank):
    if rank != 0:
        return None
    oracle, inp, cache = _oracle_setup(wl)
    threads = os.cpu_count() or 1
    bs = wl.bs
    # each step: one token of the batch (cycling), so K + W steps stay within minutes
    samples = []
    for i in range(bs):
        s = torch.zeros(bs, dtype=torch.bool)
        s[i] = True
        samples.append(s)

    def step(i):
        oracle.forward(inp, threads=threads, token_sample=samples[i % bs], expert_weights=lambda e: cache[e])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    v = args.steps / dt
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded counter-hash inputs, random-init int8 weights)",
            "config": workload_config(wl, host_alg(wl), ws),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": "one token of %s per step (its %d routed rows + shared row)" % (wl.name, wl.topk)},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_peaks():
    """Build and run the peak-rate probe (csrc/peak_probe.cu): exact-integer
    contraction rates of the two GEMM engines (dp4a, tcgen05 kind::f16 with A
    in shared or tensor memory), the legacy mma.sync s8 rate, a read-only HBM
    stream, and the K = 1024 exactness check of fp32 accumulation.  Prints
    the probe's JSON line."""
    from moe_expert_ffn_dispatch_gb300 import _build
    exe = _build.build_peak_probe()
    out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    line = out.stdout.strip().splitlines()[-1] if out.stdout.strip() else "{}"
    print(line, flush=True)
    return out.returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    # default: the largest single-GPU configuration (prefill, bs 4096); the
    # others are selectable and are also parity-test cases
    ap.add_argument("--workload", default="prefill", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-full", action="store_true",
                    help="also time one whole forward of the workload by the oracle (minutes at prefill)")
    ap.add_argument("--unfused", action="store_true",
                    help="MOE_FLAG_UNFUSED: the unfused chain (tensor-core GEMMs, separate requant and combine) "
                         "as an A/B baseline")
    ap.add_argument("--fold-routing", action="store_true",
                    help="MOE_FLAG_FOLD_ROUTING: routing weight folded into the GEMM2 row scale")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the workload's expert count (smaller cases for profiler captures)")
    ap.add_argument("--bs", type=int, default=0,
                    help="override the workload's batch size (with --experts: the same rows per expert "
                         "on fewer weights, for profiler captures)")
    ap.add_argument("--peaks", action="store_true",
                    help="build and run the peak-rate probe of this GPU instead of the benchmark")
    args = ap.parse_args()
    if args.peaks:
        sys.exit(run_peaks())
    args.warmup = max(args.warmup, 3)
    ws, rank, local = dist_env()
    wl = synth.WORKLOADS[args.workload]
    if args.experts:
        wl = synth.Workload(**{**wl.__dict__, "num_experts": args.experts, "name": "%s_e%d" % (wl.name, args.experts)})
    if args.bs:
        wl = synth.Workload(**{**wl.__dict__, "bs": args.bs, "name": "%s_bs%d" % (wl.name, args.bs)})
    if args.impl == "reference":
        res = run_reference(args, wl, ws, rank)
    else:
        res = run_ours(args, wl, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
