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


def test_barrier_count_rezeroed_after_a_reported_timeout():
    """A grid barrier that gave up can leave arrivals counted (status word 32).
    Once get_status has reported a timeout on a workspace, the handle zeroes
    that count again before the workspace's next one-launch forward, which
    must then give the same outputs as before.  The leftover count is planted
    here after a bounded debug wait ran out (no kernel is made to fail)."""
    blk, a, keep, out = _setup()
    ws = blk.workspace()
    stream = torch.cuda.current_stream()
    assert _fwd(blk, a) == m.MOE_OK
    torch.cuda.synchronize()
    ref = out.clone()
    assert m.moe_fused_debug_wait_timeout(blk.handle, ws.data_ptr(), ws.numel(), 0, stream.cuda_stream) == m.MOE_OK
    torch.cuda.synchronize()
    status = blk.region("status", workspace=ws).view(torch.int32)
    status[32] = 5  # arrivals a barrier that gave up could leave behind
    torch.cuda.synchronize()
    assert blk.status()["rc"] == m.MOE_ERR_DEVICE_TIMEOUT
    out.fill_(7.0)
    assert _fwd(blk, a) == m.MOE_OK
    torch.cuda.synchronize()
    st = blk.status()
    assert st["rc"] == m.MOE_OK and st["error_flags"] == 0, st
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert int(blk.region("status", workspace=ws).view(torch.int32)[32]) == 0
