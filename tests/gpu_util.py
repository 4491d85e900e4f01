"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded synthetic inputs and compare with the CPU oracle.

Tolerances (the block's accuracy contract):
  * integer and index work (dispatch arrays, expert_token_nums, x_q codes,
    int32 accumulators): bit-exact;
  * fp32 x_scale: bit-exact (only IEEE mul/div/max are involved);
  * SwiGLU output h: within 2e-6 relative -- the only difference between the
    two sides is the exp() implementation (CUDA expf vs the C library's expf,
    each within a few ulp);
  * requantised x2: at most 1 LSB apart on at most 0.1 % of the elements
    (an exp ulp can move a value across a rounding boundary), s2 within 2e-6;
  * bf16 (or fp16) y2 / output / share_output: bit-exact wherever the two
    sides contract the same requantised codes with the same row scale -- a
    row whose x2 and s2 equal the oracle's, a token all of whose rows do, and
    every row once the oracle's x2 / s2 are planted into the workspace (GEMM2
    dequant, FusedDeepMoE analysis §6.2, and the combine, §4.2, are fixed
    sequences of round-to-nearest fp32 operations, so nothing else may
    differ); otherwise (a row downstream of an exp-ulp code flip) per row
    max |gpu - oracle| <= 2e-2 * max |oracle row|; masked rows exactly zero.
The block is created in the workload's signature variant (x dtype, weight
scale dtype, per-expert smooth scales), the oracle reads the same inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_expert_ffn_dispatch_gb300 as m
import oracle
import synth

H_REL = 2e-6
OUT_REL = 2e-2
X2_FRAC = 1e-3
# rows of a free-running forward whose requantised codes and scale must equal
# the oracle's (and whose outputs must then be bit-exact)
MIN_EXACT_FRAC = 0.8


def device_inputs(inp, dev):
    d = {"x": inp.x.to(dev), "expert_ids": inp.expert_ids.to(dev), "expert_scales": inp.expert_scales.to(dev)}
    if inp.mask is not None:
        d["mask"] = inp.mask.to(dev)
    return d


def device_weights(inp, dev):
    w = {"w1": inp.w1.to(dev), "w1_scale": inp.w1_scale.to(dev), "w2": inp.w2.to(dev),
         "w2_scale": inp.w2_scale.to(dev)}
    if inp.wl.has_shared:
        w.update(share_w1=inp.share_w1.to(dev), share_w1_scale=inp.share_w1_scale.to(dev),
                 share_w2=inp.share_w2.to(dev), share_w2_scale=inp.share_w2_scale.to(dev))
    if inp.smooth is not None:
        w["smooth"] = inp.smooth.to(dev)
    if inp.share_smooth is not None:
        w["share_smooth"] = inp.share_smooth.to(dev)
    return w


_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "f32": torch.float32}


def make_block(wl, dev, bs_max=None, unfused=False, fold_routing=False):
    return m.MoeFused(bs_max if bs_max is not None else wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter,
                      wl.has_shared, dev, unfused=unfused, fold_routing=fold_routing,
                      act_dtype=_DT[wl.act_dtype], scale_dtype=_DT[wl.scale_dtype],
                      expert_smooth=wl.smooth_per_expert)


def region(blk, name, dtype, shape=None, workspace=None):
    t = blk.region(name, workspace=workspace).view(dtype)
    if shape is not None:
        n = int(np.prod(shape))
        t = t[:n].view(*shape)
    return t.cpu()


def assert_rows_close(got: torch.Tensor, ref: torch.Tensor, rel: float = OUT_REL, what: str = ""):
    g = got.float().cpu().double()
    r = ref.float().cpu().double()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if g.numel() == 0:
        return
    tol = rel * r.abs().amax(dim=1, keepdim=True)
    bad = (g - r).abs() > tol
    zero_rows = r.abs().amax(dim=1) == 0
    assert torch.all(g[zero_rows] == 0), "%s: rows that must be zero are not" % what
    if bad.any():
        i = int(bad.any(dim=1).nonzero()[0])
        raise AssertionError("%s: row %d max err %.3e > tol %.3e" % (what, i, float((g[i] - r[i]).abs().max()),
                                                                     float(tol[i])))


def assert_codes_close(got: torch.Tensor, ref: torch.Tensor, what: str):
    d = (got.to(torch.int32) - ref.to(torch.int32)).abs()
    if d.numel() == 0:
        return
    assert int(d.max()) <= 1, "%s: code differs by %d" % (what, int(d.max()))
    frac = float((d > 0).sum()) / d.numel()
    assert frac <= X2_FRAC, "%s: %.4f%% of codes differ" % (what, 100 * frac)


def assert_rel(got: torch.Tensor, ref: torch.Tensor, rel: float, what: str):
    g = got.double().cpu()
    r = ref.double().cpu()
    err = (g - r).abs()
    tol = rel * r.abs() + 1e-35
    if not torch.all(err <= tol):
        i = int((err - tol).argmax())
        raise AssertionError("%s: element %d got %r want %r" % (what, i, float(g.view(-1)[i]), float(r.view(-1)[i])))


SMALL_ROWS = 8  # experts with at most this many rows take the dp4a path (when h, I <= 4096)


def small_max_rows(blk, wl):
    """Largest row count of an expert (or the shared expert) that still runs on
    the dp4a path: every expert in a batch of at most 8 tokens (an expert with
    more rows, from repeated ids, in several 8-row slots), 8 otherwise; none
    with MOE_FLAG_UNFUSED or hidden / inter above 4096."""
    if not (wl.hidden <= 4096 and wl.inter <= 4096 and not (blk.cfg.flags & m.FLAG_UNFUSED)):
        return 0
    return (1 << 30) if wl.bs <= SMALL_ROWS else SMALL_ROWS


def active_tokens(inp):
    bs = inp.wl.bs
    mask = torch.ones(bs, dtype=torch.bool) if inp.mask is None else inp.mask
    return mask, mask.nonzero().view(-1)


def row_paths(blk, inp, counts):
    """Bool [rows]: GEMM rows (routed r < R, then the shared expert's rows at
    bs * topk + i) that take the tensor-core path; the others take the dp4a
    path.  An expert takes the tensor-core path when it has more than 8 rows
    (and the batch has more than 8 tokens), or always with MOE_FLAG_UNFUSED
    or when hidden or inter exceed 4096."""
    wl = inp.wl
    bs, h, K, I = wl.bs, wl.hidden, wl.topk, wl.inter
    _, act = active_tokens(inp)
    S = int(act.numel()) if wl.has_shared else 0
    rows = bs * K + (bs if wl.has_shared else 0)
    cap = small_max_rows(blk, wl)
    big = torch.zeros(rows, dtype=torch.bool)
    off = 0
    for c in counts:
        big[off:off + c] = c > cap
        off += c
    if S:
        big[bs * K:bs * K + S] = S > cap
    return big


def gpu_x2_s2(blk, inp, row_big):
    """Requantised codes and row scales of every GEMM row as the workspace
    holds them: int8 codes for dp4a rows, the exact f16 copies (x2h) for
    tensor-core rows."""
    wl = inp.wl
    rows = row_big.numel()
    I = wl.inter
    x2 = region(blk, "x2", torch.int8, (rows, I)).clone()
    x2h = region(blk, "x2h", torch.int16, (rows, I)).view(torch.float16).to(torch.int8)
    x2[row_big] = x2h[row_big]
    s2 = region(blk, "s2", torch.float32, (rows,))
    return x2, s2


def plant_x2_s2(blk, inp, ref, rows_sel=None):
    """Write the oracle's requantised codes (int8 into x2, exact f16 into x2h)
    and row scales into the workspace, for the routed rows in `rows_sel`
    (all when None) and the shared rows of those tokens."""
    wl = inp.wl
    bs, K, I = wl.bs, wl.topk, wl.inter
    R = ref["R"]
    _, act = active_tokens(inp)
    S = int(act.numel()) if wl.has_shared else 0
    rows = bs * K + (bs if wl.has_shared else 0)
    dev = blk.device
    x2v = blk.region("x2").view(torch.int8)[:rows * I].view(rows, I)
    x2hv = blk.region("x2h").view(torch.float16)[:rows * I].view(rows, I)
    s2v = blk.region("s2").view(torch.float32)[:rows]
    sel = torch.arange(R) if rows_sel is None else rows_sel
    if sel.numel():
        q = ref["x2"][sel].to(dev)
        x2v[sel.to(dev)] = q
        x2hv[sel.to(dev)] = q.to(torch.float16)
        s2v[sel.to(dev)] = ref["s2"][sel].to(dev)
    if S:
        sh = torch.arange(S) if rows_sel is None else _shared_sel(inp, ref, rows_sel)
        if sh.numel():
            q = ref["share_x2"][act[sh]].to(dev)
            idx = (bs * K + sh).to(dev)
            x2v[idx] = q
            x2hv[idx] = q.to(torch.float16)
            s2v[idx] = ref["share_s2"][act[sh]].to(dev)


def _shared_sel(inp, ref, rows_sel):
    """Indexes into the active-token list of the tokens that own `rows_sel`."""
    K = inp.wl.topk
    _, act = active_tokens(inp)
    toks = torch.unique(ref["tk_of_row"][rows_sel].long() // K)
    pos = torch.full((inp.wl.bs,), -1, dtype=torch.long)
    pos[act] = torch.arange(act.numel())
    return pos[toks][pos[toks] >= 0]


def bits(t):
    return t.contiguous().view(torch.int16)


def assert_exact_rows(blk, inp, ref, out, sout, row_big, rows_sel=None, min_frac=0.0, what=""):
    """y2 rows, outputs and shared outputs bit-exact wherever the GPU's x2 and
    s2 equal the oracle's (all of them after plant_x2_s2).  `rows_sel`
    restricts the check to those routed rows and their tokens.  Returns the
    fraction of checked rows whose inputs agreed; at least `min_frac`."""
    wl = inp.wl
    bs, h, K = wl.bs, wl.hidden, wl.topk
    R = ref["R"]
    mask, act = active_tokens(inp)
    S = int(act.numel()) if wl.has_shared else 0
    x2, s2 = gpu_x2_s2(blk, inp, row_big)
    sel = torch.arange(R) if rows_sel is None else rows_sel
    ok_r = torch.zeros(R, dtype=torch.bool)
    if sel.numel():
        ok_r[sel] = (x2[sel] == ref["x2"][sel]).all(dim=1) & (bits_f32(s2[sel]) == bits_f32(ref["s2"][sel]))
    y2 = region(blk, "y2", torch.int16, (max(R, 1), h))[:R]
    ref_y2 = bits(ref["y2"])
    okr = ok_r.nonzero().view(-1)
    assert torch.equal(y2[okr], ref_y2[okr]), "%s: y2 rows with the oracle's x2 / s2 differ" % what
    # tokens whose every dispatched row agrees (and, for the shared output, whose shared row agrees)
    toks = act if rows_sel is None else torch.unique(ref["tk_of_row"][rows_sel].long() // K)
    row_of = ref["row_of"]
    n_tok_ok = 0
    for t in toks.tolist():
        rs = [r for r in row_of[t].tolist() if r >= 0]
        if all(bool(ok_r[r]) for r in rs):
            n_tok_ok += 1
            assert torch.equal(bits(out.cpu()[t]), bits(ref["output"][t])), "%s: output token %d" % (what, t)
    n_sh, n_sh_ok = 0, 0
    if S:
        sh = torch.arange(S) if rows_sel is None else _shared_sel(inp, ref, rows_sel)
        for i in sh.tolist():
            t = int(act[i])
            n_sh += 1
            r = bs * K + i
            if torch.equal(x2[r], ref["share_x2"][t]) and \
                    bool((bits_f32(s2[r:r + 1]) == bits_f32(ref["share_s2"][t:t + 1])).all()):
                n_sh_ok += 1
                assert torch.equal(bits(sout.cpu()[t]), bits(ref["share_output"][t])), \
                    "%s: share_output token %d" % (what, t)
    checked = int(sel.numel()) + n_sh
    frac = (int(okr.numel()) + n_sh_ok) / checked if checked else 1.0
    assert frac >= min_frac, "%s: only %.3f of the rows have the oracle's x2 / s2" % (what, frac)
    return frac


def bits_f32(t):
    return t.contiguous().view(torch.int32)


def check_planted_gemm2(blk, inp, ref, di, dw, rows_sel=None, what="planted"):
    """GEMM2, its dequant and the combine on the oracle's own requantised
    codes and row scales: rerun the forward up to the requant (fresh dispatch
    and combine counters), plant the oracle's x2 / s2, run GEMM2 and the
    combine, and require y2, output and share_output bit-exact (on the rows
    and tokens of `rows_sel`, or everywhere)."""
    # one set of output tensors for both calls: the quant kernel (kernel 0)
    # zeroes the rows of masked tokens and of tokens without a valid id
    out, sout, nums = blk.forward_inputs(di, dw, until=m.KERNEL_ID["requant_big"])
    torch.cuda.synchronize()
    plant_x2_s2(blk, inp, ref, rows_sel)
    blk.forward_inputs(di, dw, start=m.KERNEL_ID["gemm2_small"], out=out, share_out=sout, token_nums=nums)
    torch.cuda.synchronize()
    st = blk.status()
    assert st["rc"] == 0 and st["error_flags"] == 0, st
    row_big = row_paths(blk, inp, ref["expert_token_nums"].tolist())
    frac = assert_exact_rows(blk, inp, ref, out, sout, row_big, rows_sel, min_frac=1.0, what=what)
    assert frac == 1.0
    return out, sout



def run_and_check(inp, dev, staged=True, bs_max=None, blk=None, planted=True):
    """Run one forward on the GPU and check every stage against the oracle;
    with `planted`, also GEMM2 and the combine on the oracle's x2 / s2, bit-exact.
    Returns (block, oracle result, (device inputs, device weights))."""
    wl = inp.wl
    bs, h, E, K, I = wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    if blk is None:
        blk = make_block(wl, dev, bs_max)
    di = device_inputs(inp, dev)
    dw = device_weights(inp, dev)
    if staged and bs > 0:
        # stop after GEMM1 (SwiGLU + requant): h is reused by y2 once GEMM2 runs
        blk.forward_inputs(di, dw, until=m.KERNEL_ID["requant_big"])
        torch.cuda.synchronize()
        staged_h = blk.region("h").clone().cpu()
    out, sout, nums = blk.forward_inputs(di, dw)
    torch.cuda.synchronize()
    st = blk.status()
    assert st["rc"] == 0 and st["error_flags"] == 0, st
    # the oracle runs in the mode the block was created in
    ref = oracle.forward(inp, intermediates=staged, threads=8,
                         fold_routing=bool(blk.cfg.flags & m.FLAG_FOLD_ROUTING))
    R = ref["R"]
    assert st["dispatched_rows"] == R
    assert st["skipped_pairs"] == ref["skipped"]
    assert torch.equal(nums.cpu(), ref["expert_token_nums"])
    mask = torch.ones(bs, dtype=torch.bool) if inp.mask is None else inp.mask
    act = mask.nonzero().view(-1)
    S = int(act.numel()) if wl.has_shared else 0
    assert st["shared_rows"] == S
    if staged and bs > 0:
        # dispatch (bit-exact)
        assert torch.equal(region(blk, "counts", torch.int32, (E,)), ref["expert_token_nums"])
        assert torch.equal(region(blk, "offsets", torch.int32, (E + 1,)), ref["offsets"])
        assert torch.equal(region(blk, "row_of", torch.int32, (bs, K)), ref["row_of"])
        assert torch.equal(region(blk, "tk_of_row", torch.int32, (R,)), ref["tk_of_row"])
        if wl.has_shared:
            assert torch.equal(region(blk, "active", torch.int32, (S,)), act.to(torch.int32))
        # quant (bit-exact on active tokens; per routed row with [E, h] smooth scales)
        per_row = inp.smooth is not None and inp.smooth.dim() == 2
        if per_row:
            xq = region(blk, "x_q", torch.int8, (R, h))
            xs = region(blk, "x_scale", torch.float32, (R,))
            assert torch.equal(xq, ref["x_q"]), "x_q (per row) differs"
            assert torch.equal(xs, ref["x_scale"]), "x_scale (per row) differs"
        else:
            xq = region(blk, "x_q", torch.int8, (bs, h))
            xs = region(blk, "x_scale", torch.float32, (bs,))
            assert torch.equal(xq[act], ref["x_q"][act]), "x_q differs"
            assert torch.equal(xs[act], ref["x_scale"][act]), "x_scale differs"
        if wl.has_shared and (inp.smooth is not None or inp.share_smooth is not None):
            assert torch.equal(region(blk, "xs_q", torch.int8, (bs, h))[act], ref["xs_q"][act])
            assert torch.equal(region(blk, "xs_scale", torch.float32, (bs,))[act], ref["xs_scale"][act])
        rows = bs * K + (bs if wl.has_shared else 0)
        # GEMM1 outputs, rows 2I floats wide: both engines leave the SwiGLU
        # output h in the first I floats of a row, fp32 within exp ulps of the
        # oracle (the dequant before it is exact: GEMM1's int32 accumulators are
        # checked bit for bit by check_raw_accumulators)
        hb = staged_h.view(torch.float32)[:rows * 2 * I].view(rows, 2 * I)
        counts = ref["expert_token_nums"].tolist()
        if R:
            assert_rel(hb[:R, :I], ref["h"], H_REL, "h routed")
        if S:
            assert_rel(hb[bs * K:bs * K + S, :I], ref["share_h"][act], H_REL, "h shared")
        # requant: dp4a rows keep int8 codes (x2); tensor-core rows keep them
        # only as exact f16 values (x2h, the tensor-core GEMM2 operand)
        x2 = region(blk, "x2", torch.int8, (rows, I)).clone()
        x2h = region(blk, "x2h", torch.int16, (rows, I)).view(torch.float16).to(torch.int8)
        row_big = row_paths(blk, inp, counts)
        x2[row_big] = x2h[row_big]
        s2 = region(blk, "s2", torch.float32, (rows,))
        assert_codes_close(x2[:R], ref["x2"], "x2 routed")
        assert_rel(s2[:R], ref["s2"], H_REL, "s2 routed")
        if S:
            assert_codes_close(x2[bs * K:bs * K + S], ref["share_x2"][act], "x2 shared")
            assert_rel(s2[bs * K:bs * K + S], ref["share_s2"][act], H_REL, "s2 shared")
        # y2 (x's dtype) of routed rows
        y2 = region(blk, "y2", torch.int16, (max(R, 1), h))[:R].view(inp.x.dtype)
        assert_rows_close(y2, ref["y2"], OUT_REL, "y2")
        # bit-exact where the requantised inputs agree (most rows: a code flips
        # only when an exp ulp moves a value across a rounding boundary)
        assert_exact_rows(blk, inp, ref, out, sout, row_big, min_frac=MIN_EXACT_FRAC, what="free-running")
    if bs > 0:
        assert out.dtype == inp.x.dtype and (sout is None or sout.dtype == inp.x.dtype)
        assert_rows_close(out, ref["output"], OUT_REL, "output")
        if wl.has_shared:
            assert_rows_close(sout, ref["share_output"], OUT_REL, "share_output")
        assert torch.all(out.cpu()[~mask].float() == 0)
    if staged and bs > 0 and planted:
        check_planted_gemm2(blk, inp, ref, di, dw)
    return blk, ref, (di, dw)


def check_raw_accumulators(blk, inp, ref, di, dw, dev):
    """int32 accumulators of both GEMMs, bit-exact.  GEMM1 runs on the x_q the
    forward left in the workspace (already checked bit-exact); for GEMM2 the
    oracle's x2 is planted into the workspace first, so both sides contract the
    same codes."""
    wl = inp.wl
    bs, h, K, I = wl.bs, wl.hidden, wl.topk, wl.inter
    R = ref["R"]
    mask = torch.ones(bs, dtype=torch.bool) if inp.mask is None else inp.mask
    act = mask.nonzero().view(-1)
    S = int(act.numel()) if wl.has_shared else 0
    rows = bs * K + (bs if wl.has_shared else 0)
    fargs = (di["x"], di["expert_ids"], di["expert_scales"], dw["w1"], dw["w1_scale"], dw["w2"], dw["w2_scale"],
             dw.get("share_w1"), dw.get("share_w1_scale"), dw.get("share_w2"), dw.get("share_w2_scale"),
             dw.get("smooth"), dw.get("share_smooth"), di.get("mask"))
    acc1 = torch.zeros(rows, 2 * I, dtype=torch.int32, device=dev)
    blk.debug_gemm_acc(1, acc1, *fargs)
    torch.cuda.synchronize()
    a1 = acc1.cpu()
    assert torch.equal(a1[:R], ref["acc1"]), "acc1 routed differs"
    if S:
        assert torch.equal(a1[bs * K:bs * K + S], ref["share_acc1"][act]), "acc1 shared differs"
    # plant the oracle's x2 (int8 for the small-expert kernel, f16 codes for the
    # tensor-core kernel) and contract it
    x2v = blk.region("x2").view(torch.int8)[:rows * I].view(rows, I)
    x2hv = blk.region("x2h").view(torch.float16)[:rows * I].view(rows, I)
    x2v[:R] = ref["x2"].to(dev)
    x2hv[:R] = ref["x2"].to(dev).to(torch.float16)
    if S:
        x2v[bs * K:bs * K + S] = ref["share_x2"][act].to(dev)
        x2hv[bs * K:bs * K + S] = ref["share_x2"][act].to(dev).to(torch.float16)
    acc2 = torch.zeros(rows, h, dtype=torch.int32, device=dev)
    blk.debug_gemm_acc(2, acc2, *fargs)
    torch.cuda.synchronize()
    a2 = acc2.cpu()
    assert torch.equal(a2[:R], ref["acc2"]), "acc2 routed differs"
    if S:
        assert torch.equal(a2[bs * K:bs * K + S], ref["share_acc2"][act]), "acc2 shared differs"
