"""Builds the CUDA library in-tree: stale_activations_gb300/_build/libdpp.so (sm_103a).

Plain nvcc, one -gencode, translation units compiled in parallel; no torch
extension machinery (the C ABI has no torch types).  build_library(bounds=True) builds
the index-checking variant (-DDPP_DEBUG_BOUNDS: every kernel checks the global indices
it computes and records the first one outside its tensor, see dpp_debug_bounds) as
_build/bounds/libdpp_bounds.so, for the tests.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libdpp.so")
BOUNDS_DIR = os.path.join(OUT_DIR, "bounds")
LIB_BOUNDS = os.path.join(BOUNDS_DIR, "libdpp_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _deps():
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
            [os.path.join(INCLUDE, "dpp.h"), os.path.abspath(__file__)])


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False, extra_flags=(),
                  bounds: bool = False) -> str:
    """Compile every csrc/*.cu and link libdpp.so (or, with bounds, the index-checking
    libdpp_bounds.so); returns its path."""
    deps = _deps()
    lib, out_dir = (LIB_BOUNDS, BOUNDS_DIR) if bounds else (LIB, OUT_DIR)
    if bounds:
        extra_flags = (*extra_flags, "-DDPP_DEBUG_BOUNDS")
    if not force and not _stale(lib, deps):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [NVCC, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        list(ex.map(compile_one, zip(srcs, objs)))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
