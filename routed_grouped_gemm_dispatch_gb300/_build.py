"""Compile the CUDA library for sm_103a (nvcc, in-tree, no cmake).

Each translation unit is compiled in parallel to an object file, then linked
into ``_build/libmoe_gb300.so``.  Rebuilds only when a source is newer than
the library.  ``build(debug=True)`` makes ``_build/libmoe_gb300_debug.so`` with
``-DMOE_DEBUG=1``: the kernels then also check their own indices, coordinates
and shared-memory layout and report a failed check as MOE_DEV_DEBUG_CHECK in
the status word (the stand-in for a sanitizer where none can run).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmoe_gb300.so")
LIB_DEBUG = os.path.join(BUILD, "libmoe_gb300_debug.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xcompiler", "-Wall", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                               + glob.glob(os.path.join(INCLUDE, "*.h")))


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    target = LIB_DEBUG if debug else LIB
    if not force and not needs_build(target):
        return target
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if debug:
        extra += ["-DMOE_DEBUG=1"]
    tag = "dbg" if debug else "rel"

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + f".{tag}.{os.getpid()}.o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, _sources()))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for _, log in results:
            print(log)
    tmp = target + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart=static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, target)
    for o in objs:
        os.remove(o)
    return target


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
