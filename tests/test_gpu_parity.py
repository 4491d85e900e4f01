"""GPU parity of the fused MoE block against the CPU oracle, through the C ABI.

Every stage is compared (see tests/gpu_util.py for the tolerances): dispatch
arrays, x_q / x_scale, int32 accumulators of both GEMMs, SwiGLU output,
requantised codes, bf16 expert rows, output and share_output -- the last three
bit-exact wherever the requantised codes agree, and everywhere once the
oracle's codes and row scales are planted before GEMM2.  Shapes span
several tiles with ragged tails: multi-block experts (> 64 rows), a partial
GEMM2 output tile (hidden % 128 == 64), a K tail (hidden % 256 != 0), one
GEMM1 tile (inter = 64), empty experts, skipped ids, masks, smooth scales.
"""
import pytest
import torch

import synth
from gpu_util import (check_planted_gemm2, check_raw_accumulators, device_inputs, device_weights, make_block,
                      region, run_and_check, small_max_rows)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None

CASES = [
    synth.WORKLOADS["tiny"],
    synth.custom("ragged_shared_mask_smooth", bs=37, hidden=192, num_experts=5, topk=3, inter=96 + 32,
                 has_shared=True, masked_fraction=0.2, smooth=True, share_smooth=True, seed=21),
    synth.custom("multi_block_experts", bs=100, hidden=320, num_experts=3, topk=2, inter=64,
                 has_shared=True, seed=22),
    synth.custom("zipf_skew", bs=64, hidden=512, num_experts=32, topk=4, inter=256, has_shared=True,
                 routing="zipf", masked_fraction=0.25, smooth=True, seed=23),
    synth.custom("topk1", bs=19, hidden=128, num_experts=4, topk=1, inter=128, has_shared=False, seed=24),
    synth.custom("balanced", bs=128, hidden=256, num_experts=16, topk=4, inter=128, has_shared=True,
                 routing="balanced", seed=25),
    synth.custom("bs1", bs=1, hidden=256, num_experts=8, topk=4, inter=128, has_shared=True, seed=26),
]


# The decode shapes' contraction lengths (hidden 4096, inter 2048): the dp4a
# GEMM1 streams K in two 2048-byte stages per weight row, the tensor-core
# GEMMs drain four (GEMM1) and two (GEMM2) exact 1024-wide accumulation
# chunks.  The int32 accumulators of both must be bit-exact there.
FULL_K_CASES = [
    # a batch of 8 tokens: every expert on the dp4a path
    synth.custom("dp4a_fullk_shared_mask_smooth", bs=8, hidden=4096, num_experts=4, topk=2, inter=2048,
                 has_shared=True, masked_fraction=0.25, smooth=True, share_smooth=True, seed=71),
    synth.custom("dp4a_fullk_plain", bs=8, hidden=4096, num_experts=4, topk=2, inter=2048, has_shared=False,
                 seed=72),
    # 40 tokens, Zipf over 8 experts: hot experts on the tensor cores, cold ones on dp4a
    synth.custom("mixed_fullk_zipf", bs=40, hidden=4096, num_experts=8, topk=2, inter=2048, has_shared=True,
                 routing="zipf", masked_fraction=0.1, smooth=True, seed=73),
    # 128 tokens over 16 experts: 6 and 7 rows on dp4a, 12-121 rows and the 128-row
    # shared expert on the tensor cores (one to two 128-row blocks)
    synth.custom("mixed_fullk_e16", bs=128, hidden=4096, num_experts=16, topk=4, inter=2048,
                 has_shared=True, routing="zipf", seed=76),
    # 160 tokens over 32 experts: 14 experts with at most 8 rows, 18 on the tensor cores
    synth.custom("mixed_fullk_e32", bs=160, hidden=4096, num_experts=32, topk=4, inter=2048, has_shared=True,
                 routing="zipf", seed=78),
]


@pytest.mark.parametrize("wl", FULL_K_CASES, ids=lambda w: w.name)
def test_full_k_staged_parity(wl):
    inp = synth.make_inputs(wl)
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True)
    counts = ref["expert_token_nums"].tolist()
    if wl.bs > 8:
        assert any(c > 8 for c in counts) and any(0 < c <= 8 for c in counts), counts
    # the slot table's split (bit-exact): experts up to the cap in slots of at
    # most 8 rows on dp4a, the others (and the shared expert above the cap) in
    # big slots on the tensor cores
    cap = small_max_rows(blk, wl)
    S = (int(inp.mask.sum()) if inp.mask is not None else wl.bs) if wl.has_shared else 0
    want_big = sum(c > cap for c in counts) + int(S > cap)
    want_small = sum((c + 7) // 8 for c in counts if 0 < c <= cap) + ((S + 7) // 8 if 0 < S <= cap else 0)
    tab = region(blk, "slots", torch.int32, (8,)).tolist()
    assert (tab[0], tab[4]) == (want_big, want_small), (tab[:8], want_big, want_small)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_staged_parity(wl):
    inp = synth.make_inputs(wl)
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


def test_all_tokens_one_expert_and_empty_experts():
    wl = synth.custom("one_expert", bs=150, hidden=256, num_experts=6, topk=1, inter=128, has_shared=True, seed=31)
    inp = synth.make_inputs(wl)
    inp.expert_ids = torch.full_like(inp.expert_ids, 4)
    blk, ref, (di, dw) = run_and_check(inp, DEV)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)
    assert ref["expert_token_nums"].tolist() == [0, 0, 0, 0, 150, 0]


def _repeated_ids_small_batch(smooth_per_expert):
    """bs 8, 4 experts, top-4 with repeated ids: 9, 9, 9 and 5 rows, so three
    experts exceed the 8-row dp4a limit and the batch needs 7 routed slots
    plus the shared one (more than E + 2)."""
    wl = synth.custom("repeated_ids_bs8" + ("_expert_smooth" if smooth_per_expert else ""), bs=8, hidden=256,
                      num_experts=4, topk=4, inter=128, has_shared=True, smooth=smooth_per_expert,
                      smooth_per_expert=smooth_per_expert, seed=34)
    inp = synth.make_inputs(wl)
    flat = torch.tensor([0] * 9 + [1] * 9 + [2] * 9 + [3] * 5, dtype=torch.int32)
    perm = synth.permutation(34, 1, flat.numel())
    inp.expert_ids = flat[perm].view(8, 4).contiguous()
    return wl, inp


@pytest.mark.parametrize("smooth_per_expert", [False, True], ids=["token_quant", "expert_smooth"])
def test_repeated_ids_in_a_small_batch_take_split_dp4a_slots(smooth_per_expert):
    """A batch of at most 8 tokens runs every expert on the dp4a path: an
    expert that repeated ids give more than 8 rows takes several slots of at
    most 8 rows, and none of the tensor-core launches (nor the separate
    combine) runs; the expand kernel runs only to quantise per routed row."""
    wl, inp = _repeated_ids_small_batch(smooth_per_expert)
    blk = make_block(wl, DEV)
    blk.set_timing(True)
    blk.get_timing()
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True, blk=blk, planted=False)
    launches = {k: n for k, (_, n) in blk.get_timing().items()}
    blk.set_timing(False)
    check_planted_gemm2(blk, inp, ref, di, dw)
    assert ref["expert_token_nums"].tolist() == [9, 9, 9, 5]
    for k in ("gemm1_big", "requant_big", "gemm2_big", "combine"):
        assert launches[k] == 0, launches
    assert (launches["expand"] > 0) == smooth_per_expert, launches
    assert launches["gemm1_small"] == 2, launches  # the staged forward and the full one
    # slot table (bit-exact): header, then seven arrays of stride E + 2 + 16;
    # experts in ascending id, each in slots of at most 8 rows, then the
    # shared expert (id -1) on its 8 active tokens after the 32 routed rows
    E, st = wl.num_experts, wl.num_experts + 2 + 16
    tab = region(blk, "slots", torch.int32, (8 + 7 * st,)).tolist()
    assert tab[0] == 0 and tab[1] == 0, tab[:8]              # no big slot, no big block
    assert tab[2] == 32 and tab[3] == 8 and tab[4] == 8, tab[:8]  # R, S, small slots
    small = tab[8 + 4 * st:]
    assert small[:8] == [0, 0, 1, 1, 2, 2, 3, -1]
    assert small[st:st + 8] == [0, 8, 9, 17, 18, 26, 27, 32]
    assert small[2 * st:2 * st + 8] == [8, 1, 8, 1, 8, 1, 5, 8]
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


def test_skipped_ids():
    wl = synth.custom("skips", bs=33, hidden=256, num_experts=8, topk=3, inter=128, has_shared=True,
                      masked_fraction=0.1, seed=32)
    inp = synth.make_inputs(wl)
    inp.expert_ids[0, 0] = -1
    inp.expert_ids[5, 2] = 8
    inp.expert_ids[7, 1] = 1 << 30
    inp.expert_ids[9, :] = -7
    run_and_check(inp, DEV)


def test_all_masked():
    wl = synth.custom("all_masked", bs=12, hidden=128, num_experts=4, topk=2, inter=64, has_shared=True, seed=33)
    inp = synth.make_inputs(wl)
    inp.mask = torch.zeros(wl.bs, dtype=torch.bool)
    blk, ref, _ = run_and_check(inp, DEV)
    assert ref["R"] == 0


def test_bs_smaller_than_bs_max_and_reused_workspace():
    """One handle and one workspace across calls with different bs and inputs:
    no state leaks from one forward into the next."""
    wl_a = synth.custom("reuse_a", bs=40, hidden=256, num_experts=8, topk=2, inter=128, has_shared=True,
                        masked_fraction=0.25, smooth=True, seed=34)
    wl_b = synth.custom("reuse_b", bs=17, hidden=256, num_experts=8, topk=2, inter=128, has_shared=True, seed=35)
    blk = make_block(wl_a, DEV, bs_max=64)
    for wl in (wl_a, wl_b, wl_a):
        inp = synth.make_inputs(wl)
        run_and_check(inp, DEV, blk=blk)


def test_bs_zero():
    wl = synth.custom("bs0", bs=0, hidden=128, num_experts=4, topk=2, inter=64, has_shared=True, seed=36)
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV, bs_max=8)
    nums = torch.full((4,), 77, dtype=torch.int32, device=DEV)
    out = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    blk.forward_inputs(device_inputs(inp, DEV), device_weights(inp, DEV), token_nums=nums, out=out,
                       share_out=torch.empty(0, 128, dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert nums.cpu().tolist() == [0, 0, 0, 0]
    assert blk.status()["dispatched_rows"] == 0


UNFUSED_CASES = [CASES[0], CASES[1], CASES[6]]


@pytest.mark.parametrize("wl", UNFUSED_CASES, ids=lambda w: w.name)
def test_unfused_chain_staged_parity(wl):
    """MOE_FLAG_UNFUSED: every expert (even with 1-8 rows) on the tensor-core
    GEMMs with the separate requant and combine kernels, against the same
    oracle and tolerances."""
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV, unfused=True)
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True, blk=blk)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


FOLD_CASES = [CASES[0], CASES[1], CASES[2], CASES[3]]


@pytest.mark.parametrize("wl", FOLD_CASES, ids=lambda w: w.name)
def test_folded_routing_staged_parity(wl):
    """MOE_FLAG_FOLD_ROUTING against the oracle's folded mode: y2 rows carry
    the routing weight, the combine is a plain sum (both GEMM paths: the
    multi-block case runs experts on the tensor cores)."""
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV, fold_routing=True)
    run_and_check(inp, DEV, staged=True, blk=blk)


def test_folded_routing_unfused_chain():
    wl = CASES[1]
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV, unfused=True, fold_routing=True)
    run_and_check(inp, DEV, staged=True, blk=blk)


def test_multi_cta_dispatch_with_masks_and_skipped_ids():
    """bs*topk = 4 * 2048 + 12: five dispatch chunks (the multi-CTA dispatch
    and its finish kernel), masked tokens, skipped ids in different chunks,
    experts spanning chunk boundaries, and experts of both GEMM paths."""
    wl = synth.custom("multi_chunk", bs=2051, hidden=128, num_experts=12, topk=4, inter=64, has_shared=True,
                      masked_fraction=0.1, smooth=True, seed=27)
    inp = synth.make_inputs(wl)
    inp.expert_ids[3, 1] = -1
    inp.expert_ids[600, 0] = 12
    inp.expert_ids[2050, 3] = 1 << 29
    inp.expert_ids[1400, :] = -3
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


# Signature variants (the operator's input table: x bf16 or fp16; routed
# weight scales fp32, bf16 or fp16; smooth scales, here per expert [E, h]):
# both GEMM paths, masks, the shared expert and a multi-block expert.
VARIANT_CASES = [
    synth.custom("fp16_bf16scale_multiblock", bs=100, hidden=320, num_experts=3, topk=2, inter=64,
                 has_shared=True, act_dtype="fp16", scale_dtype="bf16", seed=51),
    synth.custom("expert_smooth_fp16scale", bs=37, hidden=192, num_experts=5, topk=3, inter=128,
                 has_shared=True, masked_fraction=0.2, smooth=True, share_smooth=True, scale_dtype="fp16",
                 smooth_per_expert=True, seed=52),
    synth.custom("all_variants_zipf", bs=64, hidden=512, num_experts=32, topk=4, inter=256, has_shared=True,
                 routing="zipf", masked_fraction=0.25, smooth=True, act_dtype="fp16", scale_dtype="bf16",
                 smooth_per_expert=True, seed=53),
    synth.custom("expert_smooth_big_blocks", bs=300, hidden=256, num_experts=4, topk=2, inter=128,
                 has_shared=True, smooth=True, smooth_per_expert=True, seed=54),
    # more than 1216 tokens: the token quant runs one warp per token (fp16 x,
    # smooth and share-smooth scales, masked tokens' zero rows)
    synth.custom("warp_quant_fp16_smooth", bs=1300, hidden=256, num_experts=16, topk=2, inter=128,
                 has_shared=True, masked_fraction=0.3, smooth=True, share_smooth=True, act_dtype="fp16",
                 routing="zipf", seed=53),
]


@pytest.mark.parametrize("wl", VARIANT_CASES, ids=lambda w: w.name)
def test_signature_variants_staged_parity(wl):
    inp = synth.make_inputs(wl)
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


def test_signature_variants_unfused_and_folded():
    wl = VARIANT_CASES[2]
    inp = synth.make_inputs(wl)
    run_and_check(inp, DEV, staged=True, blk=make_block(wl, DEV, unfused=True))
    run_and_check(inp, DEV, staged=True, blk=make_block(wl, DEV, fold_routing=True))


# Shape limits: hidden or inter above 4096 (the dp4a path is off, every expert
# takes the tensor cores, K spans many exact 1024-wide chunks), hidden at its
# maximum (16384), 1024 experts with top-16 (most experts 0-2 rows), and a
# GEMM2 contraction of 8192.
LIMIT_CASES = [
    synth.custom("e1024_top16_h8192", bs=24, hidden=8192, num_experts=1024, topk=16, inter=64, has_shared=True,
                 masked_fraction=0.125, seed=61),
    synth.custom("hidden16384", bs=20, hidden=16384, num_experts=8, topk=4, inter=192, has_shared=True, seed=62),
    synth.custom("inter8192", bs=24, hidden=256, num_experts=4, topk=2, inter=8192, has_shared=True,
                 smooth=True, seed=63),
]


@pytest.mark.parametrize("wl", LIMIT_CASES, ids=lambda w: w.name)
def test_shape_limits_staged_parity(wl):
    inp = synth.make_inputs(wl)
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


def test_graphed_step_matches_eager_forward():
    """The captured step (one packed H2D copy, the forward, one packed D2H copy
    as one CUDA graph) gives the eager forward's outputs bit for bit, and
    picks up new inputs written into its pinned host views in place."""
    import moe_expert_ffn_dispatch_gb300 as m
    wl = CASES[3]  # zipf_skew: small and tensor-core experts, masked tokens, the shared expert
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV)
    di, dw = device_inputs(inp, DEV), device_weights(inp, DEV)
    step = m.GraphedStep(blk, {k: v.cpu() for k, v in di.items()}, dw)
    host = step.host_inputs  # the step's own pinned input views
    for trial in range(2):
        step.run()
        step.stream.synchronize()  # the step's own stream: nothing else orders it
        got = {k: v.clone() for k, v in step.host_outputs.items()}
        out, sout, nums = blk.forward_inputs({k: v.to(DEV) for k, v in host.items()}, dw)
        torch.cuda.synchronize()
        assert torch.equal(got["output"].view(torch.int16), out.cpu().view(torch.int16))
        assert torch.equal(got["share_output"].view(torch.int16), sout.cpu().view(torch.int16))
        assert torch.equal(got["expert_token_nums"], nums.cpu())
        # next step's inputs, written in place
        host["x"].copy_(torch.flip(host["x"], dims=[0]))
        host["expert_ids"].copy_(torch.roll(host["expert_ids"], 1, dims=0))


@pytest.mark.parametrize("which", ["engines_side_by_side", "one_launch"])
def test_pipelined_steps_match_eager_forward(which):
    """The pipelined serving loop (two buffer sets; the copies on their own
    streams overlap the neighbouring steps' forwards) gives every step the
    eager forward's outputs bit for bit, with new inputs written for each step
    and two steps in flight at a time.  Its CUDA graphs hold either the two
    engines side by side (a forked and joined second stream) or, for a batch
    of 8 tokens, the one-launch forward with its grid barrier."""
    import moe_expert_ffn_dispatch_gb300 as m
    if which == "one_launch":
        wl = synth.custom("pipelined_bs8", bs=8, hidden=512, num_experts=32, topk=4, inter=256, has_shared=True,
                          routing="zipf", masked_fraction=0.25, seed=96)
    else:
        wl = CASES[3]  # zipf_skew: small and tensor-core experts, masked tokens, the shared expert
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV)
    di, dw = device_inputs(inp, DEV), device_weights(inp, DEV)
    host0 = {k: v.cpu() for k, v in di.items()}
    variants = []
    for j in range(6):
        v = {k: t.clone() for k, t in host0.items()}
        v["expert_ids"] = torch.roll(v["expert_ids"], j, dims=0).contiguous()
        if j % 2:
            v["x"] = torch.flip(v["x"], dims=[0]).contiguous()
        variants.append(v)
    step = m.PipelinedStep(blk, host0, dw)
    got = []
    for k in range(0, len(variants), 2):
        for j in (k, k + 1):
            hin = step.inputs_for(j)
            for name, t in variants[j].items():
                hin[name].copy_(t)
            assert step.submit() == j
        for j in (k, k + 1):
            got.append({name: t.clone() for name, t in step.result(j).items()})
    torch.cuda.synchronize()
    for j, v in enumerate(variants):
        out, sout, nums = blk.forward_inputs({k: t.to(DEV) for k, t in v.items()}, dw)
        torch.cuda.synchronize()
        assert torch.equal(got[j]["output"].view(torch.int16), out.cpu().view(torch.int16)), j
        assert torch.equal(got[j]["share_output"].view(torch.int16), sout.cpu().view(torch.int16)), j
        assert torch.equal(got[j]["expert_token_nums"], nums.cpu()), j


def _random_cases(n=10, seed=2024):
    """Seeded random shapes within the library's limits (hidden and inter
    multiples of 64, topk <= min(E, 16)): ragged K tails, partial tiles, both
    GEMM paths, masks, smooth scales and the signature variants."""
    import random
    rng = random.Random(seed)
    out = []
    for i in range(n):
        E = rng.choice([1, 2, 3, 5, 8, 17, 40])
        topk = rng.randint(1, min(E, 16))
        per_expert = rng.random() < 0.3
        out.append(synth.custom(
            "rand%d" % i, bs=rng.choice([1, 3, 9, 31, 64, 130, 257]), hidden=64 * rng.randint(1, 12),
            num_experts=E, topk=topk, inter=64 * rng.randint(1, 10), has_shared=rng.random() < 0.7,
            routing=rng.choice(["uniform", "zipf"]) if topk < E else "uniform",
            masked_fraction=rng.choice([0.0, 0.0, 0.3]), smooth=per_expert or rng.random() < 0.4,
            share_smooth=rng.random() < 0.3, seed=300 + i, act_dtype=rng.choice(["bf16", "bf16", "fp16"]),
            scale_dtype=rng.choice(["f32", "f32", "bf16", "fp16"]), smooth_per_expert=per_expert))
    return out


@pytest.mark.parametrize("wl", _random_cases(), ids=lambda w: w.name)
def test_random_shapes_staged_parity(wl):
    inp = synth.make_inputs(wl)
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True)
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)


HALF_TILE_ROWS = [1, 8, 9, 16, 17, 32, 33, 48, 63, 64, 65, 80, 96, 128]


def test_block_row_counts_at_every_half_tile_boundary():
    """Experts with exactly 1, 8, 9, 16, 17, 32, 33, 48, 63, 64, 65, 80, 96
    and 128 rows (top-1), and a 660-row shared expert whose last block has 20:
    the tensor-core epilogues' half tiles of every size class (SwiGLU over 8
    or 16 slots a lane for halves of at most 16 / 32 rows, the 32-slot form
    above; GEMM2's chunked loop below 64 rows, its single loop at 64) staged
    against the oracle, GEMM2 and the combine bit-exact on planted codes, and
    the raw accumulators of both GEMMs."""
    bs = sum(HALF_TILE_ROWS)
    wl = synth.custom("half_tile_sizes", bs=bs, hidden=256, num_experts=len(HALF_TILE_ROWS), topk=1, inter=128,
                      has_shared=True, seed=95)
    inp = synth.make_inputs(wl)
    flat = torch.cat([torch.full((r,), e, dtype=torch.int32) for e, r in enumerate(HALF_TILE_ROWS)])
    inp.expert_ids = flat[synth.permutation(95, 1, bs)].view(bs, 1).contiguous()
    blk, ref, (di, dw) = run_and_check(inp, DEV, staged=True)
    assert ref["expert_token_nums"].tolist() == HALF_TILE_ROWS
    check_raw_accumulators(blk, inp, ref, di, dw, DEV)
