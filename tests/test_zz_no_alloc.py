"""moe_fused_dispatch_noalloc: dispatch for callers that cannot allocate.

Callers such as a plugin inside a framework that owns every device
allocation, or a process on a fixed device-memory budget, cannot hand the
library a workspace.  This entry point runs the dispatch step with its scratch
in a library-owned static device array instead.  Its outputs must equal what
the workspace-based moe_fused_forward produces for the same inputs (bit for
bit: counts and row indices are integers), on consecutive calls that reuse the
same static scratch.  This file is collected last on purpose.
"""
import pytest
import torch

import moe_expert_ffn_dispatch_gb300 as m
import synth

pytestmark = pytest.mark.gpu
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
    return nums.clone(), row_of


def _noalloc(inp, dev):
    wl = inp.wl
    ids = inp.expert_ids.to(dev)
    mask = inp.mask.to(dev).view(torch.uint8) if inp.mask is not None else None
    nums = torch.full((wl.num_experts,), -9, dtype=torch.int32, device=dev)
    rows = torch.full((wl.bs, wl.topk), -9, dtype=torch.int32, device=dev)
    rc = m.moe_fused_dispatch_noalloc(ids.data_ptr(), mask.data_ptr() if mask is not None else 0, wl.bs, wl.topk,
                                      wl.num_experts, nums.data_ptr(), rows.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == m.MOE_OK, m.moe_fused_strerror(rc)
    torch.cuda.synchronize()
    return nums, rows, (ids, mask)


def test_noalloc_dispatch_matches_forward_on_consecutive_calls():
    wl_a = synth.custom("noalloc_a", bs=96, hidden=128, num_experts=16, topk=4, inter=64, has_shared=False,
                        routing="zipf", masked_fraction=0.25, seed=51)
    wl_b = synth.custom("noalloc_b", bs=40, hidden=128, num_experts=16, topk=4, inter=64, has_shared=False, seed=52)
    inp_a, inp_b = synth.make_inputs(wl_a), synth.make_inputs(wl_b)
    inp_b.expert_ids[3, 1] = -1            # a skipped pair
    blk = m.MoeFused(96, 128, 16, 4, 64, False, DEV)
    ref_a = _forward_dispatch(blk, inp_a, DEV)
    ref_b = _forward_dispatch(blk, inp_b, DEV)
    # two calls in a row sharing the static scratch
    got_a = _noalloc(inp_a, DEV)
    got_b = _noalloc(inp_b, DEV)
    for (nums, rows, _), (rnums, rrows) in ((got_a, ref_a), (got_b, ref_b)):
        assert torch.equal(nums.cpu(), rnums.cpu())
        assert torch.equal(rows.cpu(), rrows.cpu())
    assert int(got_b[0].sum()) == wl_b.bs * wl_b.topk - 1


def test_noalloc_rejects_sizes_beyond_its_static_scratch():
    ids = torch.zeros(1, dtype=torch.int32, device=DEV)
    nums = torch.zeros(8, dtype=torch.int32, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    assert m.moe_fused_dispatch_noalloc(ids.data_ptr(), 0, 65537, 1, 8, nums.data_ptr(), 0, s) == \
        m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_fused_dispatch_noalloc(ids.data_ptr(), 0, 8, 2, 2048, nums.data_ptr(), 0, s) == \
        m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_fused_dispatch_noalloc(ids.data_ptr(), 0, 8, 2, 8, 0, 0, s) == m.MOE_ERR_INVALID_ARG
