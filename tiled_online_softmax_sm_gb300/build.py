"""Build libfa_gb300.so in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel to an object file under
``_build/`` and linked into ``libfa_gb300.so`` next to this file.  A unit is
recompiled when it, or any header it can include, is newer than its object.

``build(debug=True)`` makes ``libfa_gb300_debug.so`` instead (objects under
``_build/debug/``): the same sources with -DFA_DEBUG, whose kernels check
every global store's index against its buffer (FA_ERR_DEBUG_CHECK).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa_gb300.so")
DEBUG_LIB = os.path.join(HERE, "libfa_gb300_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


# Kernels that re-split registers with setmaxnreg: the split is sized for
# exactly this many registers per thread at launch (see the kernel source).
REQUIRED_REGS = {"fwd_bf16_kernel": 168}


def _check_regs(src: str, ptxas_log: str):
    """Refuse an object whose setmaxnreg kernels were not compiled with the
    register count their split assumes (a wrong split would stall forever)."""
    current = None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            for name, regs in REQUIRED_REGS.items():
                if name in current and int(m.group(1)) != regs:
                    raise RuntimeError(f"{src}: {name} uses {m.group(1)} registers, its "
                                       f"setmaxnreg split assumes {regs}")
            current = None


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    out_dir = os.path.join(BUILD, "debug") if debug else BUILD
    obj = os.path.join(out_dir, os.path.basename(src).replace(".cu", ".o"))
    newest = max([os.path.getmtime(src)] + [os.path.getmtime(h) for h in _headers()])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest:
        return obj
    cmd = [nvcc()] + NVCC_FLAGS + (["-DFA_DEBUG"] if debug else []) + \
        ["-Xptxas", "-v", "-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    _check_regs(src, r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    os.makedirs(os.path.join(BUILD, "debug") if debug else BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), srcs))
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
