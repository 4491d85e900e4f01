"""Host-side helpers of bench.py (no GPU): whether a committed ncu summary
still describes the current kernel code, per-forward percentiles, the clock
sampler, the algorithmic-byte accounting and the whole-forward CPU baseline."""
import os

import bench


def test_code_only_drops_comments_and_layout():
    src = ("int a = 1;  // trailing\n"
           "/* block\n   comment */ int b =\n\t2;\n")
    assert bench._code_only(src) == "int a = 1; int b = 2;"
    # a comment edit does not change the result
    assert bench._code_only(src.replace("trailing", "other words")) == bench._code_only(src)


def test_code_only_keeps_literals():
    src = 'asm volatile("{ // not a comment\\n\\t}" ::); char c = \'/\'; const char* s = "/* x */";'
    out = bench._code_only(src)
    assert '"{ // not a comment\\n\\t}"' in out
    assert "'/'" in out
    assert '"/* x */"' in out


def test_code_only_sees_code_changes():
    assert bench._code_only("x = a + b; // c") != bench._code_only("x = a - b; // c")


def test_recorded_traffic_requires_matching_sha(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    sha = bench.kernel_sha("gemm1_big")
    path = os.path.join(str(tmp_path), "gemm1_big_prefill.md")
    with open(path, "w") as f:
        f.write("traffic_bytes_per_launch: 12345\nkernel_sha: %s\n" % sha)
    assert bench.recorded_traffic("gemm1_big", "prefill") == 12345
    with open(path, "w") as f:
        f.write("traffic_bytes_per_launch: 12345\nkernel_sha: 0000000000000000\n")
    assert bench.recorded_traffic("gemm1_big", "prefill") is None
    assert bench.recorded_traffic("gemm1_big", "mid512") is None


def test_per_forward_summary_percentiles():
    s = bench.per_forward_summary([float(i) for i in range(1, 101)])  # 1 .. 100
    assert s["median"] == 50.5
    assert s["p10"] == 10.0 and s["p90"] == 90.0
    one = bench.per_forward_summary([7.0])
    assert one == {"median": 7.0, "p10": 7.0, "p90": 7.0}
    assert bench.per_forward_summary([])["median"] is None


def _fake_smi(tmp_path, body):
    d = tmp_path / "bin"
    d.mkdir()
    f = d / "nvidia-smi"
    f.write_text("#!/bin/bash\n" + body)
    f.chmod(0o755)
    return str(d)


def test_clock_sampler_starts_sampling_before_the_timed_region(tmp_path, monkeypatch):
    # a sampler that takes 0.3 s to start: entering waits for its first line
    bindir = _fake_smi(tmp_path, "sleep 0.3\nwhile true; do echo '2070, 2070, 500.0, 0x0000000000000004'; "
                                 "sleep 0.05; done\n")
    monkeypatch.setenv("PATH", bindir + os.pathsep + os.environ["PATH"])
    with bench.ClockSampler(0) as c:
        assert c.lines, "timed region would start before the first clock sample"
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] >= 1


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    with bench.ClockSampler(0) as c:
        pass
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_algorithmic_bytes_follow_the_kernel_that_runs_each_expert():
    import synth
    # bs 8: an expert with 12 rows (repeated ids) still runs in the dp4a kernels
    small_batch = synth.custom("acct8", bs=8, hidden=256, num_experts=4, topk=4, inter=128, has_shared=False)
    a = bench.algorithmic_bytes(small_batch, [12, 8, 8, 4], 8)
    assert a["gemm1_big"] == 0 and a["gemm2_big"] == 0 and a["requant_big"] == 0 and a["combine"] == 0
    assert a["gemm1_small"] > 0 and a["touched_experts"] == 4 and a["rows"] == 32
    # bs 16: the same 12-row expert takes the tensor-core kernels and the separate combine
    batch16 = synth.custom("acct16", bs=16, hidden=256, num_experts=4, topk=2, inter=128, has_shared=False)
    b = bench.algorithmic_bytes(batch16, [12, 8, 8, 4], 16)
    h, I = 256, 128
    assert b["gemm1_big"] == 2 * I * h + 8 * I + 12 * (h + 4 * I)
    assert b["combine"] > 0
    # the step total counts each touched expert's weights and scales once, plus
    # x, ids and scales, output and expert_token_nums, whichever kernels run
    w = 2 * I * h + h * I + 4 * (2 * I + h)
    assert a["step"] == 4 * w + 8 * h * 2 + 8 * 4 * 8 + 8 * h * 2 + 4 * 4
    assert b["step"] == 4 * w + 16 * h * 2 + 16 * 2 * 8 + 16 * h * 2 + 4 * 4


def test_cpu_full_forward_counts_active_tokens_of_one_whole_forward():
    """bench --cpu-full: one whole oracle forward of the workload, timed on the
    host cores, its rate over the active tokens only."""
    import synth
    wl = synth.custom("cpu_full", bs=16, hidden=128, num_experts=8, topk=2, inter=64, has_shared=True,
                      masked_fraction=0.25, seed=5)
    inp = synth.make_inputs(wl, with_weights=False)
    n_act = int(inp.mask.bool().sum())
    assert 0 < n_act < wl.bs
    r = bench.cpu_full_forward(wl)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s" and r["cores"] >= 1
    assert r["seconds"] > 0 and abs(r["value"] * r["seconds"] - n_act) < 1e-6 * n_act
    assert "one full forward of cpu_full (bs 16)" in r["sample"]
