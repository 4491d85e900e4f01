"""The oracle's pins must reject plausible mistakes.  Each case copies the
oracle source, plants one mistake (a swapped operand, a dropped term, a wrong
sign or rounding mode, an unstable dispatch ...), builds it in a temporary
directory and runs the pin suite against it in a subprocess: the suite must
fail.  Nothing here touches the real oracle build."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = [
    ("swap_gate_up",
     "float g = ((float)acc1[j] * w1s[j]) * x_scale;\n    float u = ((float)acc1[I + j] * w1s[I + j]) * x_scale;",
     "float u = ((float)acc1[j] * w1s[j]) * x_scale;\n    float g = ((float)acc1[I + j] * w1s[I + j]) * x_scale;"),
    ("exp_sign", "float t = expf(-g);", "float t = expf(g);"),
    ("truncating_cast", "float r = rintf(v);", "float r = truncf(v);"),
    ("x_scale_convention", "*scale = 1.0f / m;", "*scale = amax;"),
    ("transposed_weight",
     "const int8_t* wr = w + (size_t)n * (size_t)K;\n    int32_t s = 0;\n    for (int c = 0; c < K; ++c) s += (int32_t)a[c] * (int32_t)wr[c];",
     "int32_t s = 0;\n    for (int c = 0; c < K; ++c) s += (int32_t)a[c] * (int32_t)w[(size_t)c * N + n];"),
    ("no_amax_floor", "if (amax < ORACLE_AMAX_EPS) amax = ORACLE_AMAX_EPS;\n  float m", "float m"),
    ("combine_drops_last_k", "for (int k = 0; k < topk; ++k) {\n      if (!rows[k]) continue;",
     "for (int k = 0; k < topk - 1; ++k) {\n      if (!rows[k]) continue;"),
    ("unstable_dispatch", "int r = fill[e]++;", "int r = offsets[e + 1] - 1 - (fill[e]++ - offsets[e]);"),
    ("requant_scale", "*scale2 = amax * inv127;", "*scale2 = amax;"),
    ("shared_uses_expert_smooth", "quant_row(h, xt, a->act_fp16, a->share_smooth,",
     "quant_row(h, xt, a->act_fp16, a->smooth,"),
    ("dequant_drops_token_scale", "float g = ((float)acc1[j] * w1s[j]) * x_scale;",
     "float g = ((float)acc1[j] * w1s[j]);"),
    ("bf16_truncation", "u += 0x7FFFu + lsb;", "u += 0;"),
    ("folded_weight_dropped", "route_scale ? s2 * (*route_scale) : s2", "s2"),
    ("folded_weight_twice", "      sum = sum + act_to_f32(rows[k][c], fp16);",
     "      sum = sum + act_to_f32(rows[k][c], fp16) * 0.5f;"),
    # signature variants
    ("f16_truncation", "uint32_t q = (uint32_t)rintf(ldexpf(a, 10 - e));",
     "uint32_t q = (uint32_t)truncf(ldexpf(a, 10 - e));"),
    ("f16_subnormal_scale", "f = ldexpf((float)m, -24);", "f = ldexpf((float)m, -25);"),
    ("fp16_x_read_as_bf16", "float v = act_to_f32(x[c], fp16);", "float v = act_to_f32(x[c], 0);"),
    ("fp16_y2_written_as_bf16", "y[j] = f32_to_act(((float)acc2[j] * w2s[j]) * scale2, fp16);",
     "y[j] = f32_to_act(((float)acc2[j] * w2s[j]) * scale2, 0);"),
    ("bf16_scale_decoded_as_f16", "else if (dtype == 1) dst[i] = bf16_to_f32(",
     "else if (dtype == 1) dst[i] = f16_to_f32("),
    ("expert_smooth_wrong_row", "a->smooth + (size_t)e * h, q,", "a->smooth, q,"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, "mutation site moved: " + name
    mut = tmp_path / "moe_oracle_mutant.c"
    mut.write_text(src.replace(old, new, 1))
    env = dict(os.environ, ORACLE_MUTANT_SRC=str(mut), ORACLE_MUTANT_SO=str(tmp_path / "mutant.so"))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins accepted the mutant " + name
