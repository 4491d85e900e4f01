"""Pins for the CPU oracle: checks against closed forms, brute force, library
special cases and invariants -- never against the oracle's own formulas.

The pages print no worked numeric example, so the end-to-end floating values
are pinned by (a) an independent float64 dense evaluation with no dispatch
(brute force over (token, k) pairs) within a bound derived from the bf16
roundings, (b) exact invariants (expert relabelling, token permutation,
masking, skipped ids, topk = 1 reducing to one dense FFN), and (c) the closed
forms in tests/golden/closed_forms.json.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def f32(v):
    return np.float32(v)


def ulp32(v):
    v = abs(float(v))
    if v == 0:
        return float(np.finfo(np.float32).tiny)
    return float(np.spacing(np.float32(v)))


# ------------------------------------------------------------------ bf16
def test_bf16_rounding_matches_torch():
    """The oracle's fp32 -> bf16 cast is round-half-even: compare with torch's cast."""
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10,
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 65504.0, 3.3895e38, 0.0, -0.0],
                 dtype=np.float32),
    ])
    ours = np.array([oracle.bf16_round(float(v)) for v in vals], dtype=np.uint16)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(ours, ref)


# -------------------------------------------------------------- dispatch
def brute_dispatch(ids, E, mask):
    """Rows grouped by expert (ascending), inside a group by t then k."""
    bs, K = ids.shape
    row_of = -np.ones((bs, K), dtype=np.int64)
    tk = []
    counts = np.zeros(E, dtype=np.int64)
    for e in range(E):
        for t in range(bs):
            if mask is not None and not mask[t]:
                continue
            for k in range(K):
                if ids[t, k] == e:
                    row_of[t, k] = len(tk)
                    tk.append(t * K + k)
                    counts[e] += 1
    return counts, row_of, np.array(tk, dtype=np.int64)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dispatch_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    bs, K, E = 53, 5, 11
    ids = rng.integers(-2, E + 2, size=(bs, K)).astype(np.int32)  # some ids out of range
    mask = rng.random(bs) > 0.3
    d = oracle.dispatch(torch.from_numpy(ids), E, torch.from_numpy(mask))
    counts, row_of, tk = brute_dispatch(ids, E, mask)
    assert np.array_equal(d["counts"].numpy(), counts)
    assert np.array_equal(d["row_of"].numpy(), row_of)
    assert np.array_equal(d["tk_of_row"].numpy(), tk)
    assert np.array_equal(d["offsets"].numpy(), np.concatenate([[0], np.cumsum(counts)]))
    valid = (ids >= 0) & (ids < E) & mask[:, None]
    assert d["R"] == valid.sum() == counts.sum()
    assert d["skipped"] == ((~((ids >= 0) & (ids < E))) & mask[:, None]).sum()
    # dispatch is a permutation of the valid pairs with an exact inverse
    r = d["row_of"].numpy().reshape(-1)
    for f in range(bs * K):
        if r[f] >= 0:
            assert d["tk_of_row"][r[f]] == f


def test_dispatch_balanced_closed_form():
    """Balanced routing gives every expert exactly bs*topk/E rows."""
    wl = synth.WORKLOADS["prefill"]
    inp = synth.make_inputs(wl, with_weights=False)
    d = oracle.dispatch(inp.expert_ids, wl.num_experts)
    assert torch.all(d["counts"] == wl.bs * wl.topk // wl.num_experts)
    assert d["R"] == wl.bs * wl.topk


def test_dispatch_empty_batch():
    d = oracle.dispatch(torch.zeros(0, 4, dtype=torch.int32), 6)
    assert d["R"] == 0 and torch.all(d["counts"] == 0) and torch.all(d["offsets"] == 0)


# ----------------------------------------------------------------- quant
def test_x_quant_closed_forms(golden):
    for case in golden["x_quant"]["cases"]:
        x = torch.tensor(case["x"], dtype=torch.float32).to(torch.bfloat16)
        assert torch.equal(x.float(), torch.tensor(case["x"], dtype=torch.float32)), "input must be bf16-exact"
        sm = None if case["smooth"] is None else torch.tensor(case["smooth"], dtype=torch.float32)
        q, s = oracle.quant_row(x, sm)
        assert q.tolist() == case["q"], case["name"]
        if "scale" in case:
            assert s == case["scale"]
        if "scale_times_m" in case:
            assert abs(s * case["scale_times_m"] - 1.0) <= 2 ** -23
        if "scale_approx" in case:
            assert abs(s - case["scale_approx"]) <= 1e-6 * case["scale_approx"]


@pytest.mark.parametrize("j", [-3, 1, 5])
def test_x_quant_invariant_to_power_of_two(j):
    """Symmetric per-token quant is invariant to a positive scalar (decode case
    study, W8A8 contract); with 2**j every fp32 step scales exactly."""
    rng = np.random.default_rng(10 + j)
    x = torch.from_numpy(rng.standard_normal(512).astype(np.float32)).to(torch.bfloat16)
    q0, s0 = oracle.quant_row(x)
    q1, s1 = oracle.quant_row((x.float() * 2.0 ** j).to(torch.bfloat16))
    assert torch.equal(q0, q1)
    assert s1 == s0 * 2.0 ** j


def test_x_quant_grid_property():
    """q is the nearest grid point: |q*scale - xs| <= scale/2 (plus fp32 slack), max|q| = 127."""
    rng = np.random.default_rng(3)
    for _ in range(20):
        x = torch.from_numpy(rng.standard_normal(300).astype(np.float32) * rng.uniform(0.01, 100)).to(torch.bfloat16)
        sm = torch.from_numpy(rng.uniform(0.5, 2.0, 300).astype(np.float32))
        q, s = oracle.quant_row(x, sm)
        xs = x.double() * sm.double()
        err = (q.double() * s - xs).abs()
        assert float(err.max()) <= 0.5 * s * (1 + 1e-5)
        assert int(q.abs().max()) == 127


# -------------------------------------------------------------- requant
def test_requant_closed_forms(golden):
    inv127 = float(np.float32(1.0) / np.float32(127.0))
    for case in golden["requant"]["cases"]:
        q, s = oracle.requant_row(torch.tensor(case["h"], dtype=torch.float32))
        assert q.tolist() == case["q"], case["name"]
        if "scale_over_fp32_inv127" in case:
            assert s == case["scale_over_fp32_inv127"] * inv127


def test_requant_zero_row_and_symmetry():
    q, s = oracle.requant_row(torch.zeros(64))
    assert torch.all(q == 0)
    assert s == float(np.float32(1e-4) * (np.float32(1.0) / np.float32(127.0)))
    rng = np.random.default_rng(5)
    h = torch.from_numpy(rng.standard_normal(256).astype(np.float32) * 3)
    qa, sa = oracle.requant_row(h)
    qb, sb = oracle.requant_row(-h)
    assert torch.equal(qa, -qb) and sa == sb
    err = (qa.double() * sa - h.double()).abs()
    assert float(err.max()) <= 0.5 * sa * (1 + 1e-5)
    assert int(qa.abs().max()) == 127


# ------------------------------------------------------------------ GEMM
def test_gemm_matches_int64():
    rng = np.random.default_rng(7)
    a = rng.integers(-127, 128, size=(9, 333)).astype(np.int8)
    w = rng.integers(-128, 128, size=(45, 333)).astype(np.int8)
    ours = oracle.gemm_rows(torch.from_numpy(a), torch.from_numpy(w)).numpy()
    ref = a.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(ours.astype(np.int64), ref)


def test_gemm_closed_forms(golden):
    for case in golden["gemm"]["cases"]:
        a = torch.full((1, case["K"]), case["a"], dtype=torch.int8)
        w = torch.full((3, case["K"]), case["w"], dtype=torch.int8)
        acc = oracle.gemm_rows(a, w)
        assert torch.all(acc == case["acc"]), case["name"]


# ---------------------------------------------------------------- SwiGLU
def test_swiglu_closed_forms(golden):
    for case in golden["swiglu"]["cases"]:
        acc = torch.tensor([case["acc_gate"], case["acc_up"]], dtype=torch.int32)
        ws = torch.tensor([case["w_gate"], case["w_up"]], dtype=torch.float32)
        h = float(oracle.swiglu_row(acc, ws, case["x_scale"])[0])
        ref = case["h_exact"]
        assert abs(h - ref) <= 4 * ulp32(ref), case["name"]
        assert math.copysign(1.0, h) == math.copysign(1.0, ref), case["name"]


def test_swiglu_matches_float64():
    rng = np.random.default_rng(11)
    I = 512
    acc = rng.integers(-200000, 200000, size=2 * I).astype(np.int32)
    ws = rng.uniform(0.5, 1.5, 2 * I).astype(np.float32) / np.float32(127 * 64)
    xs = 0.021
    h = oracle.swiglu_row(torch.from_numpy(acc), torch.from_numpy(ws), xs).numpy()
    y = acc.astype(np.float64) * ws.astype(np.float64) * float(np.float32(xs))
    g, u = y[:I], y[I:]
    ref = g / (1 + np.exp(-g)) * u
    assert np.all(np.abs(h - ref) <= 8 * np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) + 1e-30)


# --------------------------------------------------------------- combine
def test_combine_closed_forms(golden):
    for case in golden["combine"]["cases"]:
        rows = [torch.tensor(r, dtype=torch.float32).to(torch.bfloat16) for r in case["rows"]]
        out = oracle.combine_token(rows, torch.tensor(case["scales"], dtype=torch.float32))
        assert out.float().tolist() == case["out"], case["name"]


def test_combine_skips_missing_rows():
    a = torch.tensor([1.0, -2.0], dtype=torch.bfloat16)
    out = oracle.combine_token([None, a, None], torch.tensor([9.0, 0.5, 9.0]))
    assert out.float().tolist() == [0.5, -1.0]


# ----------------------------------------------------------- end to end
def rne_half_even(v):
    return np.rint(v)  # numpy rint rounds half to even


def dense_reference(inp):
    """Float64 brute force: every active (token, k) pair evaluated densely with
    no dispatch, no int8 buffers shared with the oracle, no bf16 rounding of the
    expert rows.  Quant decisions are taken in float64."""
    wl = inp.wl
    bs, h, E, K, I = wl.bs, wl.hidden, wl.num_experts, wl.topk, wl.inter
    x = inp.x.double().numpy()
    ids = inp.expert_ids.numpy()
    sc = inp.expert_scales.double().numpy()
    mask = np.ones(bs, bool) if inp.mask is None else inp.mask.numpy().astype(bool)
    W1 = inp.w1.numpy().astype(np.int64)
    W2 = inp.w2.numpy().astype(np.int64)
    w1s = inp.w1_scale.double().numpy()
    w2s = inp.w2_scale.double().numpy()

    def quant(v):
        amax = max(np.abs(v).max(), 1e-4)
        s = amax / 127.0
        return np.clip(rne_half_even(v / s), -127, 127).astype(np.int64), s

    def ffn(xq, xsc, w1, s1, w2, s2):
        y1 = (w1 @ xq).astype(np.float64) * s1 * xsc
        g, u = y1[:I], y1[I:]
        hh = g / (1 + np.exp(-g)) * u
        q2, sc2 = quant(hh)
        return (w2 @ q2).astype(np.float64) * s2 * sc2

    out = np.zeros((bs, h))
    share = np.zeros((bs, h))
    sm = None if inp.smooth is None else inp.smooth.double().numpy()
    for t in range(bs):
        if not mask[t]:
            continue
        xq, xsc = quant(x[t] * (1.0 if sm is None or sm.ndim == 2 else sm))
        for k in range(K):
            e = int(ids[t, k])
            if not 0 <= e < E:
                continue
            if sm is not None and sm.ndim == 2:    # per-expert smooth: the row's own quant
                xq, xsc = quant(x[t] * sm[e])
            out[t] += sc[t, k] * ffn(xq, xsc, W1[e], w1s[e], W2[e], w2s[e])
        if wl.has_shared:
            xs2 = x[t] * (1.0 if inp.share_smooth is None else inp.share_smooth.double().numpy())
            sq, ssc = quant(xs2)
            share[t] = ffn(sq, ssc, inp.share_w1.numpy().astype(np.int64), inp.share_w1_scale.double().numpy(),
                           inp.share_w2.numpy().astype(np.int64), inp.share_w2_scale.double().numpy())
    return out, share


def rowwise_close(got, ref, rel):
    got = np.asarray(got, dtype=np.float64)
    for t in range(ref.shape[0]):
        m = np.abs(ref[t]).max()
        assert np.abs(got[t] - ref[t]).max() <= rel * m + 1e-30, (t, np.abs(got[t] - ref[t]).max(), m)


CASES = [
    synth.WORKLOADS["tiny"],
    synth.custom("ragged", bs=37, hidden=192, num_experts=5, topk=3, inter=96, has_shared=True,
                 masked_fraction=0.2, smooth=True, share_smooth=True, seed=21),
    synth.custom("zipf", bs=24, hidden=128, num_experts=16, topk=4, inter=64, has_shared=True,
                 routing="zipf", masked_fraction=0.25, smooth=True, seed=22),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_forward_matches_float64_dense(wl):
    """The relative error bound: bf16 rounding of each expert row (2^-9) and of
    the output (2^-9) over <= topk terms, plus rare one-code flips where the
    fp32 and fp64 quant decisions straddle a rounding boundary."""
    inp = synth.make_inputs(wl)
    res = oracle.forward(inp, intermediates=True, threads=4)
    ref_out, ref_share = dense_reference(inp)
    rowwise_close(res["output"].float().numpy(), ref_out, 1e-2)
    if wl.has_shared:
        rowwise_close(res["share_output"].float().numpy(), ref_share, 1e-2)
    mask = np.ones(wl.bs, bool) if inp.mask is None else inp.mask.numpy().astype(bool)
    assert np.all(res["output"].float().numpy()[~mask] == 0)
    # int32 accumulators are exact integers: compare against int64 brute force
    xq = res["x_q"].numpy().astype(np.int64)
    for r in range(res["R"]):
        f = int(res["tk_of_row"][r])
        t, e = f // wl.topk, int(inp.expert_ids.view(-1)[f])
        assert np.array_equal(res["acc1"][r].numpy(), inp.w1[e].numpy().astype(np.int64) @ xq[t])
        assert np.array_equal(res["acc2"][r].numpy(),
                              inp.w2[e].numpy().astype(np.int64) @ res["x2"][r].numpy().astype(np.int64))
    assert int(res["expert_token_nums"].sum()) == res["R"]


def test_expert_relabelling_is_exact():
    wl = CASES[1]
    inp = synth.make_inputs(wl)
    base = oracle.forward(inp, threads=4)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(wl.num_experts))
    inv = torch.argsort(perm)
    inp2 = synth.make_inputs(wl)
    inp2.expert_ids = perm[inp.expert_ids.long()].to(torch.int32)     # expert e is now called perm[e]
    inp2.w1 = inp.w1[inv].contiguous(); inp2.w2 = inp.w2[inv].contiguous()
    inp2.w1_scale = inp.w1_scale[inv].contiguous(); inp2.w2_scale = inp.w2_scale[inv].contiguous()
    res = oracle.forward(inp2, threads=4)
    assert torch.equal(res["output"].view(torch.int16), base["output"].view(torch.int16))
    assert torch.equal(res["expert_token_nums"][perm], base["expert_token_nums"])


def test_token_permutation_permutes_outputs():
    wl = CASES[2]
    inp = synth.make_inputs(wl)
    base = oracle.forward(inp, threads=4)
    p = torch.from_numpy(np.random.default_rng(2).permutation(wl.bs))
    inp.x = inp.x[p].contiguous(); inp.expert_ids = inp.expert_ids[p].contiguous()
    inp.expert_scales = inp.expert_scales[p].contiguous(); inp.mask = inp.mask[p].contiguous()
    res = oracle.forward(inp, threads=4)
    assert torch.equal(res["output"].view(torch.int16), base["output"].view(torch.int16)[p])
    assert torch.equal(res["share_output"].view(torch.int16), base["share_output"].view(torch.int16)[p])


def test_skipped_ids_equal_zero_weight():
    """A pair whose id is out of range contributes nothing: same bits as routing
    it to a real expert with expert_scale 0 (x + (+-0) = x)."""
    wl = CASES[0]
    inp = synth.make_inputs(wl)
    inp.expert_ids[3, 1] = -1
    inp.expert_ids[5, 0] = wl.num_experts + 4
    a = oracle.forward(inp, threads=2)
    assert a["skipped"] == 2 and a["R"] == wl.bs * wl.topk - 2
    inp.expert_ids[3, 1] = 0
    inp.expert_ids[5, 0] = 1
    inp.expert_scales[3, 1] = 0.0
    inp.expert_scales[5, 0] = 0.0
    b = oracle.forward(inp, threads=2)
    assert torch.equal(a["output"].view(torch.int16), b["output"].view(torch.int16))


def test_topk1_unit_scale_is_one_dense_ffn():
    """topk = 1 with expert_scale 1: the combine is the identity on the expert row,
    and the routed path equals the shared path when the shared expert has the
    same weights and smooth scales (two code paths of the oracle agree)."""
    wl = synth.custom("top1", bs=12, hidden=128, num_experts=4, topk=1, inter=64, has_shared=True,
                      smooth=True, seed=31)
    inp = synth.make_inputs(wl)
    inp.expert_scales = torch.ones_like(inp.expert_scales)
    inp.expert_ids = torch.full_like(inp.expert_ids, 2)
    inp.share_w1 = inp.w1[2].clone(); inp.share_w2 = inp.w2[2].clone()
    inp.share_w1_scale = inp.w1_scale[2].clone(); inp.share_w2_scale = inp.w2_scale[2].clone()
    inp.share_smooth = inp.smooth.clone()
    res = oracle.forward(inp, intermediates=True, threads=2)
    assert torch.equal(res["output"].view(torch.int16), res["share_output"].view(torch.int16))
    assert torch.equal(res["output"].view(torch.int16)[res["tk_of_row"].long()], res["y2"].view(torch.int16))


def test_all_masked_gives_zero_and_no_rows():
    wl = synth.custom("allmasked", bs=6, hidden=64, num_experts=3, topk=2, inter=64, has_shared=True, seed=41)
    inp = synth.make_inputs(wl)
    inp.mask = torch.zeros(wl.bs, dtype=torch.bool)
    res = oracle.forward(inp, threads=2)
    assert res["R"] == 0 and int(res["expert_token_nums"].sum()) == 0
    assert torch.all(res["output"].float() == 0) and torch.all(res["share_output"].float() == 0)


def test_token_sample_matches_full_run():
    wl = CASES[1]
    inp = synth.make_inputs(wl)
    full = oracle.forward(inp, threads=4)
    samp = torch.zeros(wl.bs, dtype=torch.bool)
    samp[torch.tensor([0, 5, 17, 36])] = True
    part = oracle.forward(inp, token_sample=samp, threads=4)
    assert torch.equal(part["output"].view(torch.int16)[samp], full["output"].view(torch.int16)[samp])
    assert torch.equal(part["share_output"].view(torch.int16)[samp], full["share_output"].view(torch.int16)[samp])


# ------------------------------------------------ folded routing weight mode
# The DeepSeek-V4 decode case study (§2.3) fuses the routing weight into the
# per-row GEMM2 dequant scale; the combine becomes a plain sum.  Pins: the
# mode equals the default mode bit for bit whenever every routing weight is a
# power of two (scaling by 2^j commutes with every rounding step), it matches
# the float64 dense evaluation within the same bound, and a dropped or
# doubled weight fails both.

def _with_scales(inp, scales):
    inp.expert_scales = scales.to(torch.float32)
    return inp


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_folded_equals_default_for_power_of_two_weights(wl):
    inp = synth.make_inputs(wl)
    g = torch.Generator().manual_seed(7)
    pw = torch.randint(-3, 2, inp.expert_scales.shape, generator=g).to(torch.float32)
    _with_scales(inp, torch.pow(2.0, pw))
    a = oracle.forward(inp, threads=4)
    b = oracle.forward(inp, threads=4, fold_routing=True)
    assert torch.equal(a["output"].view(torch.int16), b["output"].view(torch.int16))
    if wl.has_shared:
        assert torch.equal(a["share_output"].view(torch.int16), b["share_output"].view(torch.int16))


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_folded_matches_float64_dense(wl):
    inp = synth.make_inputs(wl)
    res = oracle.forward(inp, threads=4, fold_routing=True)
    ref_out, ref_share = dense_reference(inp)
    rowwise_close(res["output"].float().numpy(), ref_out, 1e-2)
    if wl.has_shared:
        rowwise_close(res["share_output"].float().numpy(), ref_share, 1e-2)


def test_folded_differs_from_default_for_generic_weights():
    # the two modes round differently (the weight multiplies before the row's
    # bf16 rounding); with softmax weights some outputs must differ
    inp = synth.make_inputs(CASES[0])
    a = oracle.forward(inp, threads=4)
    b = oracle.forward(inp, threads=4, fold_routing=True)
    assert not torch.equal(a["output"].view(torch.int16), b["output"].view(torch.int16))
    diff = (a["output"].float() - b["output"].float()).abs().max().item()
    assert diff <= 2e-2 * a["output"].float().abs().max().item()


# ------------------------------------------------------ signature variants
# The pages' input table lists x as bf16 or fp16 and the routed weight scales
# as fp32, bf16 or fp16; the smooth scales' shape is not given ([E, h] per
# expert is the variant).  Pins: the fp16 conversions against numpy's IEEE
# float16 casts (all 65536 codes one way, edge and random values the other);
# fp16 mode equal to bf16 mode through every integer stage when x is exact in
# both formats; 16-bit scales equal to their exact fp32 widening; [E, h]
# smooth equal to the [h] mode when all rows agree, and with a distinct power
# of two per expert each routed row's scale names the expert whose row it
# used; and every variant within the float64 dense bound.

def test_f16_to_f32_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_value(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))   # signed zeros too


def test_f32_to_f16_matches_numpy_rne():
    rng = np.random.default_rng(5)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
            3 * 2.0 ** -26, 2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -12), 1e-30,
            float("inf"), -float("inf"), 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0, 4097.0]
    # every f16 midpoint in a few binades (ties go to the even code)
    base = np.arange(0x3C00, 0x3C40, dtype=np.uint16).view(np.float16).astype(np.float64)
    vals += list((base[:-1] + base[1:]) / 2)
    vals += list(np.ldexp(rng.uniform(-1, 1, 4000), rng.integers(-30, 18, 4000)))
    v32 = np.array(vals, dtype=np.float32)
    ref = v32.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_round(float(v)) for v in v32], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _variant(wl, **kw):
    return synth.Workload(**{**wl.__dict__, **kw})


def test_fp16_x_equals_bf16_x_through_the_integer_stages():
    wl = CASES[1]
    inp = synth.make_inputs(wl)
    # x values with 8 significant bits and a moderate exponent: exact in both formats
    inp.x = (torch.round(inp.x.float() * 64) / 64).clamp(-3.9, 3.9).to(torch.bfloat16)
    a = oracle.forward(inp, intermediates=True, threads=4)
    inp.x = inp.x.float().to(torch.float16)
    b = oracle.forward(inp, intermediates=True, threads=4)
    for name in ("x_q", "x_scale", "acc1", "h", "x2", "s2", "acc2", "xs_q", "xs_scale", "share_acc2"):
        assert torch.equal(a[name], b[name]), name
    assert b["output"].dtype == torch.float16 and b["y2"].dtype == torch.float16
    # y2 and the outputs: one rounding of the same fp32 values, to bf16 or to fp16
    yb, yf = a["y2"].float(), b["y2"].float()
    assert ((yb - yf).abs() <= yf.abs() * 2.0 ** -8 + 1e-30).all()
    # the outputs sum topk such terms (cancellation allowed): bound by the row's largest value
    ob, of = a["output"].float(), b["output"].float()
    assert ((ob - of).abs() <= of.abs().amax(dim=1, keepdim=True) * 2.0 ** -7).all()


@pytest.mark.parametrize("sdt", ["bf16", "fp16"])
def test_16_bit_weight_scales_equal_their_fp32_widening(sdt):
    inp = synth.make_inputs(_variant(CASES[1], scale_dtype=sdt))
    assert inp.w1_scale.dtype == {"bf16": torch.bfloat16, "fp16": torch.float16}[sdt]
    a = oracle.forward(inp, threads=4)
    inp.w1_scale = inp.w1_scale.float()
    inp.w2_scale = inp.w2_scale.float()
    b = oracle.forward(inp, threads=4)
    assert torch.equal(a["output"].view(torch.int16), b["output"].view(torch.int16))
    assert torch.equal(a["share_output"].view(torch.int16), b["share_output"].view(torch.int16))


def test_per_expert_smooth_with_equal_rows_equals_vector_mode():
    wl = CASES[1]
    inp = synth.make_inputs(wl)
    a = oracle.forward(inp, threads=4)
    inp.smooth = inp.smooth.view(1, -1).repeat(wl.num_experts, 1).contiguous()
    b = oracle.forward(inp, intermediates=True, threads=4)
    assert torch.equal(a["output"].view(torch.int16), b["output"].view(torch.int16))
    assert torch.equal(a["share_output"].view(torch.int16), b["share_output"].view(torch.int16))
    assert b["x_q"].shape[0] == b["R"]


def test_per_expert_smooth_row_uses_its_own_expert():
    wl = CASES[2]
    inp = synth.make_inputs(wl)
    E, h, K = wl.num_experts, wl.hidden, wl.topk
    inp.smooth = None
    plain = oracle.forward(inp, intermediates=True, threads=4)
    j = torch.arange(E) % 5 - 2                      # expert e scales x by 2^j[e]
    inp.smooth = torch.pow(2.0, j.float()).view(E, 1).repeat(1, h).contiguous()
    res = oracle.forward(inp, intermediates=True, threads=4)
    for r in range(res["R"]):
        f = int(res["tk_of_row"][r])
        t, e = f // K, int(inp.expert_ids.view(-1)[f])
        assert torch.equal(res["x_q"][r], plain["x_q"][t])               # quant invariant to 2^j
        assert res["x_scale"][r].item() == plain["x_scale"][t].item() * 2.0 ** int(j[e])
    # same codes, so the GEMM1 accumulators equal the plain run's (the 2^j
    # stays in the row's dequant scale: smoothing is not undone later)
    assert torch.equal(res["acc1"], plain["acc1"])


VARIANT_CASES = [
    _variant(CASES[1], act_dtype="fp16", name="ragged_fp16"),
    _variant(CASES[2], scale_dtype="bf16", smooth_per_expert=True, name="zipf_bf16scale_expert_smooth"),
    _variant(CASES[1], act_dtype="fp16", scale_dtype="fp16", smooth_per_expert=True, name="ragged_all"),
]


@pytest.mark.parametrize("wl", VARIANT_CASES, ids=lambda w: w.name)
def test_variants_match_float64_dense(wl):
    inp = synth.make_inputs(wl)
    res = oracle.forward(inp, threads=4)
    ref_out, ref_share = dense_reference(inp)
    rowwise_close(res["output"].float().numpy(), ref_out, 1e-2)
    if wl.has_shared:
        rowwise_close(res["share_output"].float().numpy(), ref_share, 1e-2)
