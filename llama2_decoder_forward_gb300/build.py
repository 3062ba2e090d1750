"""Build libllama_gb300.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel to an object file;
the objects link into one shared library (CUDA runtime linked statically, the
driver's tensor-map encoder is looked up at run time, so the library loads on
machines without a GPU). Rebuilds only what is older than its sources.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libllama_gb300.so")
# The same sources with -DLLAMA_BOUNDS_CHECK=1: kernels check their shared-
# memory layouts and index invariants and flag LLAMA_FLAG_INDEX (tests only).
CHECKED_BUILD = os.path.join(BUILD, "checked")
CHECKED_LIB = os.path.join(CHECKED_BUILD, "libllama_gb300_checked.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _deps():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build_library(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile the library (checked=True: the bounds-check build) and return its path."""
    bdir, lib_path = (CHECKED_BUILD, CHECKED_LIB) if checked else (BUILD, LIB)
    extra = ["-DLLAMA_BOUNDS_CHECK=1"] if checked else []
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = _deps()
    nvcc = _nvcc()
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(bdir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + deps):
            jobs.append([nvcc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        if verbose:
            print(" ".join(cmd))
        return r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(lib_path, objs):
        run([nvcc, *ARCH, "-shared", "-o", lib_path, *objs])
    return lib_path


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
