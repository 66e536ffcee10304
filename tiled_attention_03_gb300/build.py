"""Build the CUDA library libfa.so in-tree for sm_103a (nvcc, no cmake)."""

from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfa.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC",
]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


# Debug builds (never the default; see include/fa.h): the extra compile flags and the
# file each one is built to.
DEBUG_BUILDS = {
    "serialize": (["-DFA_DEBUG_SERIALIZE"], os.path.join(PKG, "libfa_debug_serialize.so")),
    "bounds": (["-DFA_DEBUG_BOUNDS"], os.path.join(PKG, "libfa_debug_bounds.so")),
}


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build_library(force: bool = False, verbose: bool = False, debug: str | None = None) -> str:
    """Compile each translation unit in parallel, then link the shared library
    (with debug = "serialize" or "bounds": that debug build, to its own file)."""
    extra, lib = DEBUG_BUILDS[debug] if debug else ([], LIB)
    if not force and up_to_date(lib):
        return lib
    tag = f".tmp{os.getpid()}" + (f"_{debug}" if debug else "")
    objs, procs = [], []
    for src in _sources():
        obj = os.path.join(CSRC, os.path.basename(src)[:-3] + tag + ".o")
        cmd = [nvcc(), *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    failed = [p.wait() for p in procs]
    try:
        if any(failed):
            raise subprocess.CalledProcessError(max(failed), "nvcc")
        tmp = lib + tag
        cmd = [nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp]
        if verbose:
            print(" ".join(cmd))
        subprocess.check_call(cmd)
        os.replace(tmp, lib)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return lib


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
