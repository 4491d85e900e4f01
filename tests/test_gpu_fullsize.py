"""Full-size workloads (the benchmark's launch configuration) against the
oracle: dispatch arrays and x_q codes over every token, output and
share_output on a seeded sample of tokens (the oracle redraws only the
experts those tokens select), and size-independent properties."""
import pytest
import torch

import oracle
import synth
from gpu_util import assert_rows_close, device_inputs, make_block, region

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None

SAMPLE = 24


def sample_tokens(bs, seed):
    n = min(bs, SAMPLE)
    perm = synth.permutation(seed, 99, bs)[:n]
    s = torch.zeros(bs, dtype=torch.bool)
    s[perm] = True
    s[0] = True
    s[bs - 1] = True
    return s


@pytest.mark.parametrize("name", ["decode8", "decode64", "mid512", "prefill"])
def test_fullsize_sampled(name):
    wl = synth.WORKLOADS[name]
    bs, h, E, K, I = wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    inp = synth.make_inputs(wl, weight_device=DEV)
    blk = make_block(wl, DEV)
    dw = {"w1": inp.w1, "w1_scale": inp.w1_scale.to(DEV), "w2": inp.w2, "w2_scale": inp.w2_scale.to(DEV),
          "share_w1": inp.share_w1, "share_w1_scale": inp.share_w1_scale.to(DEV), "share_w2": inp.share_w2,
          "share_w2_scale": inp.share_w2_scale.to(DEV)}
    if inp.smooth is not None:
        dw["smooth"] = inp.smooth.to(DEV)
    out, sout, nums = blk.forward_inputs(device_inputs(inp, DEV), dw)
    torch.cuda.synchronize()
    st = blk.status()
    assert st["rc"] == 0 and st["error_flags"] == 0, st

    # dispatch over every token (bit-exact)
    d = oracle.dispatch(inp.expert_ids, E, inp.mask)
    assert torch.equal(nums.cpu(), d["counts"])
    assert torch.equal(region(blk, "row_of", torch.int32, (bs, K)), d["row_of"])
    assert torch.equal(region(blk, "tk_of_row", torch.int32, (d["R"],)), d["tk_of_row"])
    mask = torch.ones(bs, dtype=torch.bool) if inp.mask is None else inp.mask
    assert int(nums.sum()) == int(mask.sum()) * K == st["dispatched_rows"]
    if name == "prefill":
        assert torch.all(nums == bs * K // E)

    # x_q codes and scales over every active token (bit-exact)
    xq = region(blk, "x_q", torch.int8, (bs, h))
    xs = region(blk, "x_scale", torch.float32, (bs,))
    for t in mask.nonzero().view(-1).tolist():
        q, s = oracle.quant_row(inp.x[t], inp.smooth)
        assert torch.equal(xq[t], q), t
        assert xs[t].item() == s, t

    # outputs on a sample of tokens
    samp = sample_tokens(bs, wl.seed) & mask
    ref = oracle.forward(inp, token_sample=samp,
                         expert_weights=lambda e: (synth.draw_w1(wl, e), synth.draw_w2(wl, e)))
    idx = samp.nonzero().view(-1)
    assert_rows_close(out.cpu()[idx], ref["output"][idx], what="output")
    assert_rows_close(sout.cpu()[idx], ref["share_output"][idx], what="share_output")
    assert torch.all(out.cpu()[~mask].float() == 0) and torch.all(sout.cpu()[~mask].float() == 0)
