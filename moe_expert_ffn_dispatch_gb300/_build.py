"""Build the CUDA library in-tree with nvcc for sm_103a (one -gencode).

Translation units compile in parallel; the shared object lands next to this
file as _moe_fused.so.  The host side links only the CUDA runtime.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(HERE, "_moe_fused.so")
SOURCES = ["api.cu", "dispatch_quant.cu", "moe_gemm.cu", "tc_gemm.cu"]
HEADERS = ["device_prims.cuh", "epilogue_ops.cuh", "moe_internal.h", "quant_ops.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-fmad=false",            # every fp32 step rounds once; kernels also use explicit _rn intrinsics
    "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "moe_fused.h"), __file__]
    flags = NVCC_FLAGS + list(extra_flags or [])
    procs, objs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if _stale(o, [s] + hdrs):
            cmd = [nvcc()] + flags + ["-I", INCLUDE, "-I", CSRC, "-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        msg = "\n".join("%s:\n%s" % f for f in failed)
        raise RuntimeError("nvcc failed\n" + msg)
    if _stale(SO, objs):
        tmp = SO + ".%d.tmp" % os.getpid()
        cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp] + objs + ["-lcudart"]
        subprocess.check_call(cmd)
        os.replace(tmp, SO)
    return SO


def build_peak_probe(verbose: bool = False) -> str:
    """The standalone peak-rate probe (csrc/peak_probe.cu), used by
    `bench.py --peaks`; not part of the library."""
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(CSRC, "peak_probe.cu")
    exe = os.path.join(BUILD, "peak_probe")
    if _stale(exe, [src] + [os.path.join(CSRC, h) for h in HEADERS]):
        cmd = [nvcc()] + NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC, src, "-o", exe]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
    return exe


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
