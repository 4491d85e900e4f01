"""Host-side helpers of bench.py that decide whether a committed ncu summary
still describes the current kernel code (no GPU)."""
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
