"""Host-side argument checks of the C ABI on a GPU machine: each bad call returns
its error code before any launch and leaves the outputs untouched."""
import pytest
import torch

import moe_expert_ffn_dispatch_gb300 as m
import synth
from gpu_util import device_inputs, device_weights, make_block

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _setup():
    wl = synth.custom("errs", bs=8, hidden=128, num_experts=4, topk=2, inter=64, has_shared=True, seed=41)
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV)
    di, dw = device_inputs(inp, DEV), device_weights(inp, DEV)
    out = torch.full((8, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    a, keep, _ = blk.make_args(di["x"], di["expert_ids"], di["expert_scales"], dw["w1"], dw["w1_scale"], dw["w2"],
                               dw["w2_scale"], dw["share_w1"], dw["share_w1_scale"], dw["share_w2"],
                               dw["share_w2_scale"], out=out)
    return blk, a, keep, out


def _fwd(blk, a, ws=None, nbytes=None):
    w = blk.workspace() if ws is None else ws
    return m.moe_fused_forward(blk.handle, a, w.data_ptr(), w.numel() if nbytes is None else nbytes,
                               torch.cuda.current_stream().cuda_stream)


def test_error_codes_leave_outputs_untouched():
    blk, a, keep, out = _setup()
    assert _fwd(blk, a, nbytes=blk.workspace_bytes - 1) == m.MOE_ERR_WORKSPACE_TOO_SMALL
    a.bs = 9
    assert _fwd(blk, a) == m.MOE_ERR_UNSUPPORTED_SHAPE
    a.bs = 8
    x = a.x
    a.x = x + 2
    assert _fwd(blk, a) == m.MOE_ERR_ALIGNMENT
    a.x = 0
    assert _fwd(blk, a) == m.MOE_ERR_INVALID_ARG
    a.x = x
    sw = a.share_gmm1_weight
    a.share_gmm1_weight = 0
    assert _fwd(blk, a) == m.MOE_ERR_INVALID_ARG
    a.share_gmm1_weight = sw
    ws = blk.workspace()
    assert _fwd(blk, a, ws=ws[16:], nbytes=blk.workspace_bytes) == m.MOE_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert torch.all(out.float().cpu() == 3.0)
    assert _fwd(blk, a) == m.MOE_OK
    torch.cuda.synchronize()
    assert not torch.all(out.float().cpu() == 3.0)


def test_create_rejects_bad_config():
    bad = [m.Config(8, 100, 4, 2, 64, 0, 0), m.Config(8, 128, 4, 5, 64, 0, 0), m.Config(8, 128, 0, 1, 64, 0, 0),
           m.Config(8, 128, 4, 2, 64, 0, 64), m.Config(-1, 128, 4, 2, 64, 0, 0),
           m.Config(8, 128, 4, 2, 64, 0, m.FLAG_SCALE_BF16 | m.FLAG_SCALE_FP16)]  # bit 6 reserved; one scale dtype
    for cfg in bad:
        rc, h, _ = m.moe_fused_create(cfg)
        assert rc < 0 and h == 0


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "flag"])
def test_bounded_wait_runs_out_and_reports(which):
    """A wait that nothing satisfies gives up after its 2 s budget and reports
    through the status word (no fault, no trap); the context stays usable and
    the next forward clears the status."""
    import time
    blk, a, keep, out = _setup()
    ws = blk.workspace()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert m.moe_fused_debug_wait_timeout(blk.handle, ws.data_ptr(), ws.numel(), which, stream.cuda_stream) == m.MOE_OK
    st = blk.status()
    elapsed = time.perf_counter() - t0
    assert st["rc"] == m.MOE_ERR_DEVICE_TIMEOUT
    assert st["error_flags"] & 1
    assert st["error_site"] == m.DEBUG_WAIT_SITE + which
    assert 1.5 < elapsed < 30.0
    assert m.moe_fused_debug_wait_timeout(blk.handle, ws.data_ptr(), ws.numel(), 2, stream.cuda_stream) == \
        m.MOE_ERR_INVALID_ARG
    assert _fwd(blk, a) == m.MOE_OK
    torch.cuda.synchronize()
    st = blk.status()
    assert st["rc"] == m.MOE_OK and st["error_flags"] == 0


def _plant(t, gen):
    """Overwrite a workspace region (a CUDA byte tensor) with seeded garbage."""
    t.copy_(torch.randint(0, 256, (t.numel(),), generator=gen, dtype=torch.uint8).to(t.device))


def test_one_launch_barrier_needs_no_initial_state():
    """The one-launch forward's grid barrier (its generation and per-CTA
    arrival tags) and the status words 32..47 may hold anything when a
    forward starts, e.g. memory that held other data at an address the
    handle has seen before: outputs stay bit-equal and no wait runs out."""
    blk, a, keep, out = _setup()
    ws = blk.workspace()
    assert _fwd(blk, a) == m.MOE_OK
    torch.cuda.synchronize()
    assert blk.status()["rc"] == m.MOE_OK
    ref = out.clone()
    gen = torch.Generator().manual_seed(71)
    tags = blk.region("bar_tags", workspace=ws)
    words = blk.region("status", workspace=ws)[128:192]
    for pattern in ("random", "next_generation", "ones"):
        if pattern == "random":
            _plant(tags, gen)
        elif pattern == "next_generation":  # every tag equal to the unsalted next generation
            t64 = tags.view(torch.int64)
            t64[1:] = t64[0] + 1
        else:
            tags.fill_(0xFF)
        _plant(words, gen)
        torch.cuda.synchronize()
        out.fill_(7.0)
        assert _fwd(blk, a) == m.MOE_OK
        torch.cuda.synchronize()
        st = blk.status()
        assert st["rc"] == m.MOE_OK and st["error_flags"] == 0, (pattern, st)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), pattern


def test_side_by_side_counters_need_no_initial_state():
    """The arrival counters of the side-by-side launches (status words
    40..42) are zeroed by each forward's dispatch: garbage planted there
    between forwards changes nothing."""
    wl = synth.custom("errs_split", bs=40, hidden=256, num_experts=32, topk=4, inter=192, has_shared=True,
                      routing="zipf", seed=92)
    inp = synth.make_inputs(wl)
    blk = make_block(wl, DEV)
    di, dw = device_inputs(inp, DEV), device_weights(inp, DEV)
    ws = blk.workspace()
    ref = blk.forward_inputs(di, dw)
    torch.cuda.synchronize()
    st = blk.status()
    assert st["rc"] == m.MOE_OK and st["error_flags"] == 0, st
    slots = blk.region("slots", workspace=ws).view(torch.int32)
    assert int(slots[6]) == 1 and 0 < int(slots[5]) < min(torch.cuda.get_device_properties(DEV).multi_processor_count,
                                                          1023), slots[:8]   # both engines had work
    gen = torch.Generator().manual_seed(72)
    words = blk.region("status", workspace=ws)[128:192]
    for _ in range(2):
        _plant(words, gen)
        torch.cuda.synchronize()
        got = blk.forward_inputs(di, dw)
        torch.cuda.synchronize()
        st = blk.status()
        assert st["rc"] == m.MOE_OK and st["error_flags"] == 0, st
        for x, y in zip(ref, got):
            assert torch.equal(x.view(torch.int16) if x.dtype != torch.int32 else x,
                               y.view(torch.int16) if y.dtype != torch.int32 else y)
