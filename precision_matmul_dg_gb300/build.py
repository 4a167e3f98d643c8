"""Builds libdg.so in-tree with nvcc for sm_103a (GB300).

Usage:  python -m precision_matmul_dg_gb300.build   (or __graft_entry__.build())

Each translation unit compiles in its own nvcc process (in parallel), then
one nvcc link produces precision_matmul_dg_gb300/libdg.so with the CUDA
runtime linked statically.  Objects go to precision_matmul_dg_gb300/_build/.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdg.so")

SOURCES = ["api.cu", "planner.cpp", "gemv.cu", "gemm_tc.cu", "gemm_conv.cu", "widen.cu",
           "skinny.cu", "mx.cu", "gemm_w4t.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I", INCLUDE, "-I", CSRC]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _compile(src, verbose_ptxas=False):
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + ARCH + COMMON
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    if src.endswith(".cpp"):
        cmd += ["-x", "cu"]  # host-only C++, compiled through nvcc for one toolchain
    cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def _stale(objs):
    if not os.path.exists(LIB):
        return True
    lib_t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dg.h")]
    return any(os.path.getmtime(d) > lib_t for d in deps)


def build(force=False, verbose_ptxas=False, quiet=True):
    """Compile libdg.so if any source is newer than it.  Returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    if not force and not _stale(None):
        return LIB
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    failed = [r for r in results if r[2] != 0]
    for src, _, rc, out in results:
        if out.strip() and (not quiet or rc != 0 or verbose_ptxas):
            sys.stderr.write("---- %s ----\n%s\n" % (src, out))
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(r[0] for r in failed))
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + [r[1] for r in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, quiet=False)
    print(LIB)
