"""The one-launch forward of a batch of at most 8 tokens (dispatch, quant,
GEMM1, GEMM2 and combine in one persistent launch) against the two-launch
forward of the same block (the dispatch + quant launch, then the streamed
GEMM launch) on the same inputs.

The one-launch kernel repeats, per CTA, the dispatch kernel's counting sort,
slot table and item split, and runs the same token quant, so every output
and every intermediate the two forwards leave in their workspaces must be
equal bit for bit.  The one-launch workspace starts filled with a byte
pattern, so a region it failed to write shows, and its grid-barrier words
start as garbage (the library zeroes the arrival count on a workspace's
first use).  Two one-launch forwards on different inputs run back to back
on that workspace (the barrier's state carries over).  Outputs are also
checked against the oracle: dispatch bit-exact, outputs within the
free-running tolerance of gpu_util.
"""
import copy

import pytest
import torch

import moe_expert_ffn_dispatch_gb300 as m
import oracle
import synth
from gpu_util import assert_rows_close, device_inputs, device_weights, make_block, region

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _skip_ids(inp, seed, n):
    """Plant ids outside [0, E) at seeded positions (pairs the dispatch skips)."""
    flat = inp.expert_ids.view(-1)
    pos = synth.permutation(seed, 5, flat.numel())[:n]
    for i, v in zip(pos.tolist(), (-1, inp.wl.num_experts, 1 << 20, -5)):
        flat[i] = v


def _repeated_ids(wl):
    inp = synth.make_inputs(wl)
    flat = torch.tensor([0] * 9 + [1] * 9 + [2] * 9 + [3] * 5, dtype=torch.int32)
    inp.expert_ids = flat[synth.permutation(wl.seed, 1, flat.numel())].view(8, 4).contiguous()
    return inp


def _case(name):
    c = synth.custom
    if name == "tiny":
        return synth.make_inputs(synth.WORKLOADS["tiny"]), False
    if name == "shared_mask_smooth_skips":
        wl = c(name, bs=8, hidden=512, num_experts=64, topk=8, inter=256, has_shared=True, masked_fraction=0.25,
               smooth=True, share_smooth=True, seed=81)
        inp = synth.make_inputs(wl)
        _skip_ids(inp, 81, 4)
        return inp, False
    if name == "one_token":
        return synth.make_inputs(c(name, bs=1, hidden=256, num_experts=32, topk=4, inter=128, has_shared=True,
                                   seed=82)), False
    if name == "fp16_bf16scale_folded":
        return synth.make_inputs(c(name, bs=5, hidden=256, num_experts=16, topk=4, inter=192, has_shared=True,
                                   act_dtype="fp16", scale_dtype="bf16", routing="zipf", seed=83)), True
    if name == "all_masked":
        inp = synth.make_inputs(c(name, bs=3, hidden=128, num_experts=8, topk=2, inter=64, has_shared=True,
                                  seed=84))
        inp.mask = torch.zeros(3, dtype=torch.bool)
        return inp, False
    if name == "e1024_top16":
        return synth.make_inputs(c(name, bs=8, hidden=128, num_experts=1024, topk=16, inter=64, has_shared=True,
                                   seed=85)), False
    if name == "repeated_ids":
        return _repeated_ids(c(name, bs=8, hidden=256, num_experts=4, topk=4, inter=128, has_shared=True,
                               seed=86)), False
    raise KeyError(name)


CASES = ["tiny", "shared_mask_smooth_skips", "one_token", "fp16_bf16scale_folded", "all_masked", "e1024_top16",
         "repeated_ids"]


def _two_launch(blk, di, dw):
    """dispatch + quant launch, then the streamed GEMM launch, on the block's own workspace."""
    out, sout, nums = blk.forward_inputs(di, dw, until=m.KERNEL_ID["dispatch_quant"])
    blk.forward_inputs(di, dw, start=m.KERNEL_ID["gemm1_small"], out=out, share_out=sout, token_nums=nums)
    torch.cuda.synchronize()
    return out, sout, nums


def _regions(blk, ws, inp, dw):
    """Every intermediate a forward of this batch defines, as CPU tensors."""
    wl = inp.wl
    bs, h, E, K, I = wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    i32, f32 = torch.int32, torch.float32
    st = region(blk, "status", i32, (64,), workspace=ws)
    R, S_sh, ns = int(st[3]), int(st[4]), int(st[5])
    mask = torch.ones(bs, dtype=torch.bool) if inp.mask is None else inp.mask
    act = mask.nonzero().view(-1)
    rows = list(range(R)) + list(range(bs * K, bs * K + S_sh))
    G = min(torch.cuda.get_device_properties(DEV).multi_processor_count, 1023)
    stride = E + 2 + 16
    slots = region(blk, "slots", i32, (8 + 7 * stride,), workspace=ws)
    ranges = region(blk, "ranges", i32, (2 * 1024,), workspace=ws)
    d = {
        "status": st[:6],
        "counts": region(blk, "counts", i32, (E,), workspace=ws),
        "offsets": region(blk, "offsets", i32, (E + 1,), workspace=ws),
        "row_of": region(blk, "row_of", i32, (bs * K,), workspace=ws),
        "tk_of_row": region(blk, "tk_of_row", i32, (bs * K,), workspace=ws)[:R],
        "active": region(blk, "active", i32, (bs,), workspace=ws)[:act.numel()],
        "row_token": region(blk, "row_token", i32, (bs * K + bs,) if wl.has_shared else (bs * K,),
                            workspace=ws)[rows],
        "slot_header": slots[:5],
        "big_block_prefix": slots[8 + 3 * stride:8 + 3 * stride + 1],
        "small_slots": torch.stack([slots[8 + (4 + j) * stride:8 + (4 + j) * stride + ns] for j in range(3)]),
        "ranges": torch.cat([ranges[:G + 1], ranges[1024:1024 + G + 1]]),
        "blk_ticket": blk.region("blk_ticket", workspace=ws).view(i32).cpu(),
        "tok_ticket": region(blk, "tok_ticket", i32, (bs,), workspace=ws),
        "tok_expect": region(blk, "tok_expect", i32, (bs,), workspace=ws),
        "x_q": region(blk, "x_q", torch.int8, (bs, h), workspace=ws)[act],
        "x_scale": region(blk, "x_scale", f32, (bs,), workspace=ws)[act],
        "h": region(blk, "h", f32, (bs * K + (bs if wl.has_shared else 0), 2 * I), workspace=ws)[rows, :I],
        "x2": region(blk, "x2", torch.int8, (bs * K + (bs if wl.has_shared else 0), I), workspace=ws)[rows],
        "s2": region(blk, "s2", f32, (bs * K + (bs if wl.has_shared else 0),), workspace=ws)[rows],
        "y2": region(blk, "y2", torch.int16, (bs * K, h), workspace=ws)[:R],
    }
    if wl.has_shared:
        d["shared_row"] = region(blk, "shared_row", i32, (bs,), workspace=ws)
        if dw.get("smooth") is not dw.get("share_smooth"):  # the shared expert has its own quant
            d["xs_q"] = region(blk, "xs_q", torch.int8, (bs, h), workspace=ws)[act]
            d["xs_scale"] = region(blk, "xs_scale", f32, (bs,), workspace=ws)[act]
    return d


def _bits(t):
    if t is None:
        return None
    return t.view(torch.int16).cpu() if t.dtype in (torch.bfloat16, torch.float16) else t.cpu()


def _assert_same(a, b, what):
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.float32:
            x, y = x.view(torch.int32), y.view(torch.int32)
        assert torch.equal(x, y), f"{what}: {k} differs between the one-launch and the two-launch forward"


@pytest.mark.parametrize("name", CASES)
def test_one_launch_equals_two_launch_and_oracle(name):
    inp, folded = _case(name)
    wl = inp.wl
    # a second batch for the same block: new tokens, ids, routing weights and mask
    nxt = synth.make_inputs(synth.custom(wl.name + "_next", bs=wl.bs, hidden=wl.hidden, num_experts=wl.num_experts,
                                         topk=wl.topk, inter=wl.inter, has_shared=wl.has_shared, routing="zipf",
                                         masked_fraction=0.25 if wl.bs > 1 else 0.0, seed=wl.seed + 500,
                                         act_dtype=wl.act_dtype, scale_dtype=wl.scale_dtype), with_weights=False)
    inp2 = copy.copy(inp)
    inp2.x, inp2.expert_ids, inp2.expert_scales, inp2.mask = nxt.x, nxt.expert_ids, nxt.expert_scales, nxt.mask
    blk = make_block(wl, DEV, fold_routing=folded)
    dw = device_weights(inp, DEV)
    ws1 = blk.workspace()
    raw = torch.full((blk.workspace_bytes + 256,), 0x5A, dtype=torch.uint8, device=DEV)
    ws2 = blk._aligned(raw)
    blk.set_timing(True)
    blk.get_timing()
    for step, cur in enumerate((inp, inp2)):
        di = device_inputs(cur, DEV)
        cur_w = dw
        ref_out = _two_launch(blk, di, cur_w)
        ref_reg = _regions(blk, ws1, cur, cur_w)
        out, sout, nums = blk.forward_inputs(di, cur_w, workspace=ws2)
        torch.cuda.synchronize()
        st = blk.status(workspace=ws2)
        assert st["rc"] == 0 and st["error_flags"] == 0, st
        what = f"{name} step {step}"
        for a, b in zip(ref_out, (out, sout, nums)):
            assert (a is None) == (b is None)
            if a is not None:
                assert torch.equal(_bits(a), _bits(b)), f"{what}: outputs differ"
        _assert_same(ref_reg, _regions(blk, ws2, cur, cur_w), what)
        # and the oracle
        ref = oracle.forward(cur, intermediates=False, threads=8, fold_routing=folded)
        assert torch.equal(nums.cpu(), ref["expert_token_nums"])
        assert st["skipped_pairs"] == ref["skipped"] and st["dispatched_rows"] == ref["R"]
        assert_rows_close(out.cpu(), ref["output"], what=what + " output")
        if wl.has_shared:
            assert_rows_close(sout.cpu(), ref["share_output"], what=what + " share_output")
    launches = {k: n for k, (_, n) in blk.get_timing().items()}
    blk.set_timing(False)
    # two-launch forwards: dispatch_quant + gemm1_small each; one-launch: gemm1_small only
    assert launches["dispatch_quant"] == 2 and launches["gemm1_small"] == 4, launches
    for k in ("dispatch_finish", "expand", "gemm1_big", "requant_big", "gemm2_small", "gemm2_big", "combine"):
        assert launches[k] == 0, launches
