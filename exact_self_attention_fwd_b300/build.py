"""Build the CUDA library in-tree for sm_103a (nvcc cross-compiles; no GPU needed).

    python -m exact_self_attention_fwd_b300.build [--verbose]

produces exact_self_attention_fwd_b300/libattn_fwd.so. The CUDA runtime is linked
statically, and the driver's tensor-map encoder is looked up at run time, so the
library loads on a machine without a GPU driver (calls then report ATTN_ERR_CUDA).
"""
from __future__ import annotations

import argparse
import os
import re
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libattn_fwd.so")
DEBUG_LIB = os.path.join(PKG, "libattn_fwd_debug.so")  # index-checked build (ATTN_DEBUG)
SOURCES = [os.path.join(CSRC, "attn_fwd.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "attn_bwd.cuh"),
                  os.path.join(INCLUDE, "attn_api.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(p) <= t for p in DEPS)


def _split_constants() -> dict:
    src = open(SOURCES[0]).read()
    out = {}
    for name in ("NUM_THREADS", "LAUNCH_REGS", "PRODUCER_REGS", "SOFTMAX_REGS"):
        m = re.search(rf"constexpr int {name} = (\d+);", src)
        out[name] = int(m.group(1))
    return out


def check_registers(ptxas_log: str, allow_spills: bool = False) -> None:
    """The forward kernels launch at a fixed register count and then move registers
    between warpgroups with setmaxnreg; the split must fit in the launch allocation
    and nothing may spill (the index-checked debug build may). Refuse the build
    otherwise."""
    k = _split_constants()
    need = 2 * 128 * k["SOFTMAX_REGS"] + 128 * k["PRODUCER_REGS"]
    blocks = re.split(r"Compiling entry function", ptxas_log)
    seen = 0
    for blk in blocks[1:]:
        head = blk.split("\n", 1)[0]
        if "attn_bwd_kernel" in head:
            spill = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", blk)
            if spill and (int(spill.group(1)) or int(spill.group(2))) and not allow_spills:
                raise RuntimeError("backward kernel spills registers:\n" + blk)
            continue
        if "attn_fwd_kernel" not in head:
            continue
        seen += 1
        regs = int(re.search(r"Used (\d+) registers", blk).group(1))
        spill = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", blk)
        if regs * k["NUM_THREADS"] < need:
            raise RuntimeError(f"register split {need} exceeds launch allocation {regs} x {k['NUM_THREADS']}")
        if spill and (int(spill.group(1)) or int(spill.group(2))) and not allow_spills:
            raise RuntimeError("forward kernel spills registers:\n" + blk)
    if seen == 0:
        raise RuntimeError("ptxas output did not list the forward kernels")


def build(force: bool = False, verbose: bool = False, out: str | None = None, debug: bool = False) -> str:
    """Compile the library (or, debug=True, its index-checked build) in-tree."""
    out = out or (DEBUG_LIB if debug else LIB)
    if not force and up_to_date(out):
        return out
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "static", "-I", INCLUDE, "-I", CSRC, "-o", out + ".tmp", *SOURCES]
    if debug:
        cmd += ["-DATTN_DEBUG"]
    cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    check_registers(res.stdout + res.stderr, allow_spills=debug)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the index-checked build (libattn_fwd_debug.so)")
    a = ap.parse_args()
    print(build(force=a.force or a.verbose, verbose=a.verbose, debug=a.debug))
