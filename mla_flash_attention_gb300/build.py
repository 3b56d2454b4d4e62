"""Build the C-ABI shared library ``libmla_gb300.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel, then the objects are
linked into one shared library next to this file.  No cmake, no torch extension
machinery: the library has a plain C interface (include/mla.h).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmla_gb300.so")
# the bounds-checked build (-DMLA_DEBUG): every output, LSE and workspace store is checked
# against its buffer on the device; load it by pointing MLA_GB300_LIB at it
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libmla_gb300_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: %s\n%s\n%s" % (" ".join(cmd), r.stdout, r.stderr))
    return r.stdout + r.stderr


def build(verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    """Compile every csrc/*.cu and link libmla_gb300.so (debug: the bounds-checked
    libmla_gb300_debug.so); returns the library path."""
    bdir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug:
        extra += ["-DMLA_DEBUG"]
    nv = nvcc()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        out = _run([nv, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj])
        return obj, out

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for _, out in results:
            if out.strip():
                sys.stdout.write(out)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp"
    _run([nv, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv, debug="--debug" in sys.argv))
