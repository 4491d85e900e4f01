"""Full-size workloads (the benchmark's launch configuration) against the
oracle.  decode8, decode64 and mid512 are checked on every active token;
prefill on a seeded sample of 256 tokens (the oracle redraws only the experts
the checked tokens select, from the same seeded generator):
  * dispatch arrays, expert_token_nums and x_q codes over every token
    (bit-exact);
  * free-running outputs within 2e-2 per row, and bit-exact on every checked
    token whose requantised codes and row scales equal the oracle's;
  * GEMM1 int32 accumulators of the checked tokens' rows (bit-exact);
  * requantised codes within 1 LSB on at most 0.1 %, row scales within 2e-6;
  * with the oracle's codes and row scales planted before GEMM2: GEMM2 int32
    accumulators, y2 rows, output and share_output bit-exact.
"""
import pytest
import torch

import oracle
import synth
from gpu_util import (MIN_EXACT_FRAC, H_REL, _shared_sel, active_tokens, assert_codes_close, assert_exact_rows,
                      assert_rel, assert_rows_close, check_planted_gemm2, device_inputs, gpu_x2_s2, make_block,
                      region, row_paths)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None

# tokens checked against the oracle: every active token, except at prefill
SAMPLE = {"prefill": 256}


def checked_tokens(name, bs, seed, mask):
    if name not in SAMPLE:
        return mask.clone()
    perm = synth.permutation(seed, 99, bs)[:SAMPLE[name]]
    s = torch.zeros(bs, dtype=torch.bool)
    s[perm] = True
    s[0] = True
    s[bs - 1] = True
    return s & mask


def gemm_acc(blk, which, n_cols, di, dw, rows):
    acc = torch.zeros(rows, n_cols, dtype=torch.int32, device=DEV)
    blk.debug_gemm_acc(which, acc, di["x"], di["expert_ids"], di["expert_scales"], dw["w1"], dw["w1_scale"],
                       dw["w2"], dw["w2_scale"], dw.get("share_w1"), dw.get("share_w1_scale"), dw.get("share_w2"),
                       dw.get("share_w2_scale"), dw.get("smooth"), dw.get("share_smooth"), di.get("mask"))
    torch.cuda.synchronize()
    return acc.cpu()


@pytest.mark.parametrize("name", ["decode8", "decode64", "mid512", "prefill"])
def test_fullsize(name):
    wl = synth.WORKLOADS[name]
    bs, h, E, K, I = wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    inp = synth.make_inputs(wl, weight_device=DEV)
    blk = make_block(wl, DEV)
    dw = {"w1": inp.w1, "w1_scale": inp.w1_scale.to(DEV), "w2": inp.w2, "w2_scale": inp.w2_scale.to(DEV),
          "share_w1": inp.share_w1, "share_w1_scale": inp.share_w1_scale.to(DEV), "share_w2": inp.share_w2,
          "share_w2_scale": inp.share_w2_scale.to(DEV)}
    if inp.smooth is not None:
        dw["smooth"] = inp.smooth.to(DEV)
    di = device_inputs(inp, DEV)
    out, sout, nums = blk.forward_inputs(di, dw)
    torch.cuda.synchronize()
    st = blk.status()
    assert st["rc"] == 0 and st["error_flags"] == 0, st

    # dispatch over every token (bit-exact)
    d = oracle.dispatch(inp.expert_ids, E, inp.mask)
    assert torch.equal(nums.cpu(), d["counts"])
    assert torch.equal(region(blk, "row_of", torch.int32, (bs, K)), d["row_of"])
    assert torch.equal(region(blk, "tk_of_row", torch.int32, (d["R"],)), d["tk_of_row"])
    mask, act = active_tokens(inp)
    assert int(nums.sum()) == int(mask.sum()) * K == st["dispatched_rows"]
    if name == "prefill":
        assert torch.all(nums == bs * K // E)

    # x_q codes and scales over every active token (bit-exact)
    xq = region(blk, "x_q", torch.int8, (bs, h))
    xs = region(blk, "x_scale", torch.float32, (bs,))
    for t in act.tolist():
        q, s = oracle.quant_row(inp.x[t], inp.smooth)
        assert torch.equal(xq[t], q), t
        assert xs[t].item() == s, t

    # the oracle on the checked tokens
    samp = checked_tokens(name, bs, wl.seed, mask)
    full = bool(torch.equal(samp, mask))
    ref = oracle.forward(inp, intermediates=True, token_sample=None if full else samp,
                         expert_weights=lambda e: (synth.draw_w1(wl, e), synth.draw_w2(wl, e)))
    R = ref["R"]
    tok_of_row = ref["tk_of_row"].long() // K
    rows_sel = samp[tok_of_row].nonzero().view(-1)
    sh = _shared_sel(inp, ref, rows_sel)
    rows = bs * K + bs
    idx = samp.nonzero().view(-1)
    assert idx.numel() > 0

    # free-running outputs: within 2e-2 per row, bit-exact where the codes agree
    assert_rows_close(out.cpu()[idx], ref["output"][idx], what="output")
    assert_rows_close(sout.cpu()[idx], ref["share_output"][idx], what="share_output")
    assert torch.all(out.cpu()[~mask].float() == 0) and torch.all(sout.cpu()[~mask].float() == 0)
    row_big = row_paths(blk, inp, d["counts"].tolist())
    assert_exact_rows(blk, inp, ref, out, sout, row_big, rows_sel, min_frac=MIN_EXACT_FRAC, what=name)
    x2, s2 = gpu_x2_s2(blk, inp, row_big)
    assert_codes_close(x2[rows_sel], ref["x2"][rows_sel], "x2 routed")
    assert_rel(s2[rows_sel], ref["s2"][rows_sel], H_REL, "s2 routed")
    assert_codes_close(x2[bs * K + sh], ref["share_x2"][act[sh]], "x2 shared")
    assert_rel(s2[bs * K + sh], ref["share_s2"][act[sh]], H_REL, "s2 shared")

    # GEMM1 int32 accumulators of the checked rows (on the forward's x_q)
    acc1 = gemm_acc(blk, 1, 2 * I, di, dw, rows)
    assert torch.equal(acc1[rows_sel], ref["acc1"][rows_sel]), "acc1 routed"
    assert torch.equal(acc1[bs * K + sh], ref["share_acc1"][act[sh]]), "acc1 shared"
    del acc1

    # GEMM2 and the combine on the oracle's codes and row scales: bit-exact
    check_planted_gemm2(blk, inp, ref, di, dw, rows_sel=None if full else rows_sel, what=name + " planted")
    acc2 = gemm_acc(blk, 2, h, di, dw, rows)
    assert torch.equal(acc2[rows_sel], ref["acc2"][rows_sel]), "acc2 routed"
    assert torch.equal(acc2[bs * K + sh], ref["share_acc2"][act[sh]]), "acc2 shared"
