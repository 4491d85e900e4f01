"""moe_fused_dispatch_noalloc: dispatch for callers that cannot allocate.

Callers such as a plugin inside a framework that owns every device
allocation, or a process on a fixed device-memory budget, cannot hand the
library a workspace.  This entry point runs the dispatch step with its scratch
in a library-owned static device array instead.  Its outputs are integers, so
they must equal the CPU oracle's dispatch bit for bit (counts, and the row of
every (t, k) pair in expert-sorted order, -1 where a pair is not dispatched),
and equal what the workspace-based moe_fused_forward writes for the same
inputs.  The calls below run back to back and share the one static scratch
array, up to the entry point's stated limits (bs * topk = 65536 pairs, 1024
experts, top-16).  This file is collected last on purpose: a run that stops at
its first failure has then already run every other test.
"""
import pytest
import torch

import moe_expert_ffn_dispatch_gb300 as m
import oracle
import synth

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _forward_dispatch(blk, inp, dev):
    di = {"x": inp.x.to(dev), "expert_ids": inp.expert_ids.to(dev), "expert_scales": inp.expert_scales.to(dev)}
    if inp.mask is not None:
        di["mask"] = inp.mask.to(dev)
    wl = inp.wl
    w = {"w1": inp.w1.to(dev), "w1_scale": inp.w1_scale.to(dev), "w2": inp.w2.to(dev),
         "w2_scale": inp.w2_scale.to(dev)}
    _, _, nums = blk.forward_inputs(di, w)
    torch.cuda.synchronize()
    n = wl.bs * wl.topk
    row_of = blk.region("row_of").view(torch.int32)[:n].view(wl.bs, wl.topk).clone()
    return nums.cpu(), row_of.cpu()


def _noalloc(ids_cpu, mask_cpu, E, dev):
    bs, topk = ids_cpu.shape
    ids = ids_cpu.to(dev)
    mask = mask_cpu.to(dev).view(torch.uint8) if mask_cpu is not None else None
    nums = torch.full((E,), -9, dtype=torch.int32, device=dev)
    rows = torch.full((bs, topk), -9, dtype=torch.int32, device=dev)
    rc = m.moe_fused_dispatch_noalloc(ids.data_ptr(), mask.data_ptr() if mask is not None else 0, bs, topk, E,
                                      nums.data_ptr(), rows.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == m.MOE_OK, m.moe_fused_strerror(rc)
    torch.cuda.synchronize()
    return nums.cpu(), rows.cpu()


def _assert_matches_oracle(got, ids, mask, E):
    nums, rows = got
    ref = oracle.dispatch(ids, E, mask)
    assert torch.equal(nums, ref["counts"]), "expert_token_nums differs from the oracle"
    assert torch.equal(rows, ref["row_of"]), "expand_row differs from the oracle"
    return ref


def _ids_with_skips(ids, seed):
    """Plant ids outside [0, E) (skipped pairs) at seeded positions."""
    ids = ids.clone()
    flat = ids.view(-1)
    pos = synth.permutation(seed, 7, flat.numel())[:5]
    for i, v in zip(pos.tolist(), (-1, -7, 1 << 30, 1 << 20, -(1 << 30))):
        flat[i] = v
    return ids


@pytest.mark.gpu
def test_noalloc_dispatch_matches_forward_and_oracle_on_consecutive_calls():
    wl_a = synth.custom("noalloc_a", bs=96, hidden=128, num_experts=16, topk=4, inter=64, has_shared=False,
                        routing="zipf", masked_fraction=0.25, seed=51)
    wl_b = synth.custom("noalloc_b", bs=40, hidden=128, num_experts=16, topk=4, inter=64, has_shared=False, seed=52)
    inp_a, inp_b = synth.make_inputs(wl_a), synth.make_inputs(wl_b)
    inp_b.expert_ids[3, 1] = -1            # a skipped pair
    blk = m.MoeFused(96, 128, 16, 4, 64, False, DEV)
    ref_a = _forward_dispatch(blk, inp_a, DEV)
    ref_b = _forward_dispatch(blk, inp_b, DEV)
    # two calls in a row sharing the static scratch
    got_a = _noalloc(inp_a.expert_ids, inp_a.mask, 16, DEV)
    got_b = _noalloc(inp_b.expert_ids, inp_b.mask, 16, DEV)
    for got, ref, inp in ((got_a, ref_a, inp_a), (got_b, ref_b, inp_b)):
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        _assert_matches_oracle(got, inp.expert_ids, inp.mask, 16)
    assert int(got_b[0].sum()) == wl_b.bs * wl_b.topk - 1


@pytest.mark.gpu
def test_noalloc_at_its_limits_matches_oracle():
    """65536 pairs with 1024 experts (Zipf routing, a quarter of the tokens
    masked, skipped ids), then 65536 pairs at top-16 over 1024 experts, then a
    small batch again: three consecutive calls on the shared static scratch,
    each bit-exact against the oracle."""
    wl1 = synth.custom("noalloc_limit_zipf", bs=8192, hidden=64, num_experts=1024, topk=8, inter=64,
                       routing="zipf", masked_fraction=0.25, seed=61)
    inp1 = synth.make_inputs(wl1, with_weights=False)
    ids1 = _ids_with_skips(inp1.expert_ids, 61)
    wl2 = synth.custom("noalloc_limit_top16", bs=4096, hidden=64, num_experts=1024, topk=16, inter=64, seed=62)
    inp2 = synth.make_inputs(wl2, with_weights=False)
    wl3 = synth.custom("noalloc_after_limits", bs=5, hidden=64, num_experts=1024, topk=16, inter=64,
                       routing="zipf", seed=63)
    inp3 = synth.make_inputs(wl3, with_weights=False)
    ref1 = _assert_matches_oracle(_noalloc(ids1, inp1.mask, 1024, DEV), ids1, inp1.mask, 1024)
    assert ref1["skipped"] > 0 and ref1["R"] < wl1.bs * wl1.topk
    ref2 = _assert_matches_oracle(_noalloc(inp2.expert_ids, None, 1024, DEV), inp2.expert_ids, None, 1024)
    assert ref2["R"] == 65536
    _assert_matches_oracle(_noalloc(inp3.expert_ids, None, 1024, DEV), inp3.expert_ids, None, 1024)


@pytest.mark.gpu
def test_noalloc_above_the_forward_single_cta_limit():
    """8200 pairs: the forward dispatches this many with its multi-CTA kernels,
    the no-alloc entry with its one CTA; both must give the oracle's arrays."""
    wl = synth.custom("noalloc_8200", bs=1025, hidden=64, num_experts=64, topk=8, inter=64, has_shared=False,
                      routing="zipf", masked_fraction=0.1, seed=64)
    inp = synth.make_inputs(wl)
    blk = m.MoeFused(wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter, False, DEV)
    fwd = _forward_dispatch(blk, inp, DEV)
    got = _noalloc(inp.expert_ids, inp.mask, wl.num_experts, DEV)
    _assert_matches_oracle(got, inp.expert_ids, inp.mask, wl.num_experts)
    assert torch.equal(got[0], fwd[0]) and torch.equal(got[1], fwd[1])


def test_noalloc_rejects_bad_arguments_before_any_launch():
    """Host-side checks return before any CUDA call, so they hold without a
    GPU: sizes beyond the static scratch, a NULL output, and int32 pointers
    that are not 4-byte aligned (the kernel reads ids and writes counts as
    int32 words; such a pointer would fault on the GPU)."""
    s = 0
    good = 1 << 20  # a 256-byte aligned stand-in address; nothing dereferences it
    assert m.moe_fused_dispatch_noalloc(good, 0, 65537, 1, 8, good, 0, s) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_fused_dispatch_noalloc(good, 0, 4097, 16, 1024, good, 0, s) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_fused_dispatch_noalloc(good, 0, 8, 2, 2048, good, 0, s) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_fused_dispatch_noalloc(good, 0, 8, 17, 32, good, 0, s) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_fused_dispatch_noalloc(good, 0, 8, 2, 8, 0, 0, s) == m.MOE_ERR_INVALID_ARG
    assert m.moe_fused_dispatch_noalloc(0, 0, 8, 2, 8, good, 0, s) == m.MOE_ERR_INVALID_ARG
    assert m.moe_fused_dispatch_noalloc(good + 2, 0, 8, 2, 8, good, 0, s) == m.MOE_ERR_ALIGNMENT
    assert m.moe_fused_dispatch_noalloc(good, 0, 8, 2, 8, good + 1, 0, s) == m.MOE_ERR_ALIGNMENT
    assert m.moe_fused_dispatch_noalloc(good, 0, 8, 2, 8, good, good + 2, s) == m.MOE_ERR_ALIGNMENT
