"""Build libkvq.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each .cu under csrc/ compiles to an object in parallel; the objects link into
quantized_kv_decode_gb300/libkvq.so.  Run ``python -m quantized_kv_decode_gb300.build``.
``--debug`` (build(debug=True)) compiles the same sources with KVQ_DEBUG into
libkvq_debug.so: every global access of the kernels is checked against the
extent of its array first (see kvq_debug_checks in include/kvq.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvq.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libkvq_debug.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH = "-gencode=arch=compute_103a,code=sm_103a"
# Hidden default visibility: the library exports its C ABI (KVQ_API in
# include/kvq.h) and nothing else, so that two builds loaded in one process
# (release and debug) share no C++ symbol, in particular no function-local
# static of a template (GCC would make those process-wide unique symbols).
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", ARCH, "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        [os.path.join(INCLUDE, "kvq.h"), os.path.abspath(__file__)]


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    """Compile csrc/*.cu into libkvq.so (debug: libkvq_debug.so, with the
    bounds checks of KVQ_DEBUG); returns the library path."""
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and up_to_date(debug):
        return lib
    nvcc = _nvcc()
    os.makedirs(bdir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DKVQ_DEBUG"] if debug else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    for src, _, r in results:
        if verbose or ptxas_info or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
    tmp = lib + ".tmp"
    cmd = [nvcc, ARCH, "-shared", "-o", tmp, *[o for _, o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
