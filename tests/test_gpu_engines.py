"""The two GEMM engines side by side: in a whole forward of a batch of more
than 8 tokens, the dp4a launch (experts with at most 8 rows) and the
tensor-core chain (GEMM1, requant, GEMM2 of the others) run at the same time
on disjoint CTA sets, split by the dispatch; each launch's CTAs take their
work in arrival order.  The same forward run as a sequence of kernels on one
stream (a forward stopped before the combine, then the combine) must leave
the same outputs and intermediates bit for bit, whatever the split: both
engines compute every row in the same fixed order however many CTAs they
have.  Outputs are also checked against the oracle.
"""
import pytest
import torch

import moe_expert_ffn_dispatch_gb300 as m
import oracle
import synth
from gpu_util import assert_rows_close, device_inputs, device_weights, make_block, region

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _case(name):
    c = synth.custom
    if name == "mixed_zipf_shared":    # hot experts on the tensor cores, the rest on dp4a
        return c(name, bs=64, hidden=512, num_experts=64, topk=8, inter=256, has_shared=True, routing="zipf",
                 masked_fraction=0.25, smooth=True, seed=91), "mixed"
    if name == "mixed_fp16_folded":
        return c(name, bs=40, hidden=256, num_experts=32, topk=4, inter=192, has_shared=True, routing="zipf",
                 act_dtype="fp16", scale_dtype="bf16", share_smooth=True, seed=92), "mixed"
    if name == "no_small_work":        # every expert above 8 rows
        return c(name, bs=256, hidden=256, num_experts=16, topk=4, inter=128, has_shared=True,
                 routing="balanced", seed=93), "big_only"
    if name == "no_big_work":          # no shared expert, every routed expert at most 8 rows
        return c(name, bs=16, hidden=256, num_experts=256, topk=2, inter=128, has_shared=False, seed=94), "small_only"
    raise KeyError(name)


CASES = ["mixed_zipf_shared", "mixed_fp16_folded", "no_small_work", "no_big_work"]


def _sequential(blk, di, dw):
    """The forward as kernels in sequence on one stream: up to GEMM2, then the combine."""
    out, sout, nums = blk.forward_inputs(di, dw, until=m.KERNEL_ID["gemm2_big"])
    blk.forward_inputs(di, dw, start=m.KERNEL_ID["combine"], out=out, share_out=sout, token_nums=nums)
    torch.cuda.synchronize()
    return out, sout, nums


def _slot_rows(blk, ws, E):
    """Rows of the small slots and of the big slots, from the slot table."""
    st = E + 2 + 16
    tab = region(blk, "slots", torch.int32, (8 + 7 * st,), workspace=ws).tolist()
    small = [r for i in range(tab[4]) for r in range(tab[8 + 5 * st + i], tab[8 + 5 * st + i] + tab[8 + 6 * st + i])]
    big = [r for i in range(tab[0]) for r in range(tab[8 + st + i], tab[8 + st + i] + tab[8 + 2 * st + i])]
    return small, big


def _state(blk, ws, wl, R, S):
    """What the forward defines: h of every row; the requantised codes as int8
    (dp4a rows) or as the f16 GEMM2 operand (tensor-core rows), s2; y2."""
    bs, h, E, K, I = wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    rows = bs * K + (bs if wl.has_shared else 0)
    used = list(range(R)) + list(range(bs * K, bs * K + S))  # routed rows, then the active tokens' shared rows
    small, big = _slot_rows(blk, ws, E)
    assert sorted(small + big) == used
    return {
        "row_of": region(blk, "row_of", torch.int32, (bs * K,), workspace=ws),
        "h": region(blk, "h", torch.float32, (rows, 2 * I), workspace=ws)[used, :I].view(torch.int32),
        "x2": region(blk, "x2", torch.int8, (rows, I), workspace=ws)[small],
        "x2h": region(blk, "x2h", torch.int16, (rows, I), workspace=ws)[big],
        "s2": region(blk, "s2", torch.float32, (rows,), workspace=ws)[used].view(torch.int32),
        "y2": region(blk, "y2", torch.int16, (bs * K, h), workspace=ws)[:R],
    }


def _bits(t):
    return None if t is None else t.view(torch.int16).cpu() if t.dtype in (torch.bfloat16, torch.float16) else t.cpu()


@pytest.mark.parametrize("name", CASES)
def test_engines_side_by_side_equal_the_sequential_forward(name):
    wl, kind = _case(name)
    folded = name.endswith("folded")
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV, fold_routing=folded)
    di, dw = device_inputs(inp, DEV), device_weights(inp, DEV)
    ref_out = _sequential(blk, di, dw)
    st_seq = blk.status()
    assert st_seq["rc"] == 0 and st_seq["error_flags"] == 0, st_seq
    R, S = st_seq["dispatched_rows"], st_seq["shared_rows"]
    ref_state = _state(blk, blk.workspace(), wl, R, S)
    seq_slots = region(blk, "slots", torch.int32, (8,))
    G = min(torch.cuda.get_device_properties(DEV).multi_processor_count, 1023)
    assert seq_slots[5] == G and seq_slots[6] == 0, seq_slots       # one engine after the other
    ws2 = blk._aligned(torch.full((blk.workspace_bytes + 256,), 0x3C, dtype=torch.uint8, device=DEV))
    for rep in range(2):  # twice: the arrival counters return to zero after each launch
        out, sout, nums = blk.forward_inputs(di, dw, workspace=ws2)
        torch.cuda.synchronize()
        st = blk.status(workspace=ws2)
        assert st["rc"] == 0 and st["error_flags"] == 0, (rep, st)
        for a, b in zip(ref_out, (out, sout, nums)):
            assert (a is None) == (b is None)
            if a is not None:
                assert torch.equal(_bits(a), _bits(b)), f"{name} rep {rep}: outputs differ from the sequential forward"
        got = _state(blk, ws2, wl, R, S)
        for k in ref_state:
            assert torch.equal(ref_state[k], got[k]), f"{name} rep {rep}: {k} differs from the sequential forward"
        slots = region(blk, "slots", torch.int32, (8,), workspace=ws2)
        assert slots[6] == 1, slots
        if kind == "mixed":
            assert 0 < slots[5] < G, slots
        elif kind == "big_only":
            assert slots[5] == 0 and slots[4] == 0, slots
        else:
            assert slots[5] == G and slots[1] == 0, slots
        status = region(blk, "status", torch.int32, (64,), workspace=ws2)
        assert status[40:43].tolist() == [0, 0, 0], status[40:43]   # arrival counters back at zero
    ref = oracle.forward(inp, intermediates=False, threads=8, fold_routing=folded)
    assert torch.equal(nums.cpu(), ref["expert_token_nums"])
    assert_rows_close(out.cpu(), ref["output"], what=name + " output")
    if wl.has_shared:
        assert_rows_close(sout.cpu(), ref["share_output"], what=name + " share_output")
