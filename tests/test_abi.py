"""The C-ABI library loads and exports every entry point the header declares;
struct layouts agree between the header (compiled with gcc) and the Python
binding; host-only entry points behave without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import moe_expert_ffn_dispatch_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_fused.h")


@pytest.fixture(scope="module")
def built():
    from moe_expert_ffn_dispatch_gb300 import _build
    _build.build()
    return m.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_fused_\w+)\s*\(", src)))


def test_exports_match_header(built):
    decl = declared_functions()
    assert decl, "no declarations found"
    assert sorted(m.EXPORTS) == decl
    out = subprocess.run(["nm", "-D", "--defined-only", m.LIB_PATH], capture_output=True, text=True).stdout
    syms = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in decl:
        assert name in syms, name
        getattr(built, name)


def test_struct_layout_matches_header(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text('''#include <stdio.h>
#include <stddef.h>
#include "moe_fused.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(moe_fused_config_t), sizeof(moe_fused_args_t),
         sizeof(moe_fused_status_t), offsetof(moe_fused_args_t, bs), offsetof(moe_fused_args_t, output),
         offsetof(moe_fused_args_t, x_active_mask));
  return 0; }
''')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    vals = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    assert vals == [ctypes.sizeof(m.Config), ctypes.sizeof(m.Args), ctypes.sizeof(m.Status),
                    m.Args.bs.offset, m.Args.output.offset, m.Args.x_active_mask.offset]


def test_workspace_size_and_config_checks(built):
    rc, nb = m.moe_fused_workspace_size(m.Config(4096, 4096, 256, 8, 2048, 1, 0))
    assert rc == 0
    rows = 4096 * 9
    assert nb >= rows * 2048 * 4 + rows * 2048 + 2 * 4096 * 4096
    assert nb % 256 == 0
    for cfg, code in [(m.Config(8, 100, 4, 2, 64, 0, 0), m.MOE_ERR_UNSUPPORTED_SHAPE),
                      (m.Config(8, 128, 4, 5, 64, 0, 0), m.MOE_ERR_UNSUPPORTED_SHAPE),
                      (m.Config(8, 128, 4, 2, 64, 0, 64), m.MOE_ERR_INVALID_ARG),  # reserved flag bit
                      (m.Config(8, 128, 4, 2, 64, 0, m.FLAG_SCALE_BF16 | m.FLAG_SCALE_FP16),
                       m.MOE_ERR_INVALID_ARG),  # two scale dtypes
                      (m.Config(8, 128, 2000, 2, 64, 0, 0), m.MOE_ERR_UNSUPPORTED_SHAPE),
                      (m.Config(8, 128, 4, 2, 64, 2, 0), m.MOE_ERR_INVALID_ARG)]:
        assert m.moe_fused_workspace_size(cfg)[0] == code
    for flags in (m.FLAG_UNFUSED, m.FLAG_FOLD_ROUTING, m.FLAG_UNFUSED | m.FLAG_FOLD_ROUTING, m.FLAG_FP16_ACT,
                  m.FLAG_SCALE_BF16, m.FLAG_SCALE_FP16 | m.FLAG_EXPERT_SMOOTH, 63 & ~m.FLAG_SCALE_FP16):
        assert m.moe_fused_workspace_size(m.Config(8, 128, 4, 2, 64, 0, flags))[0] == m.MOE_OK
    # per-expert smooth scales quantise every routed pair on its own: x_q grows to bs * topk rows
    base = m.moe_fused_workspace_size(m.Config(64, 4096, 256, 8, 2048, 1, 0))[1]
    per_row = m.moe_fused_workspace_size(m.Config(64, 4096, 256, 8, 2048, 1, m.FLAG_EXPERT_SMOOTH))[1]
    assert per_row - base >= 64 * 7 * 4096


def test_strerror_and_names(built):
    assert m.moe_fused_strerror(0) == "ok"
    assert "workspace" in m.moe_fused_strerror(m.MOE_ERR_WORKSPACE_TOO_SMALL)
    assert [m.moe_fused_kernel_name(k) for k in range(len(m.KERNEL_NAMES))] == m.KERNEL_NAMES
    assert m.moe_fused_destroy(0) == 0
