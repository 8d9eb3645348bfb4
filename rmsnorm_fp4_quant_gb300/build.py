"""Builds libfp4q.so in-tree (rmsnorm_fp4_quant_gb300/lib/) with nvcc for sm_103a.

Each .cu under csrc/ is compiled to an object in parallel, then linked into
one shared library with the CUDA runtime linked statically, so the library
loads on any machine with a driver and no matching libcudart.  Rebuilds only
when a source or header is newer than the library.

With --debug (or build(debug=True)) the same sources are compiled with
-DFP4Q_DEBUG_CHECKS into libfp4q_debug.so: every computed global address is
checked against its buffer's extent and a fault injector for the bounded waits
is compiled in (include/fp4q.h, "Debug build").

    python -m rmsnorm_fp4_quant_gb300.build [--force] [--verbose] [--debug]
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIBNAME = "libfp4q.so"
LIBPATH = os.path.join(LIBDIR, LIBNAME)
DEBUG_LIBPATH = os.path.join(LIBDIR, "libfp4q_debug.so")
DEBUG_FLAGS = ["-DFP4Q_DEBUG_CHECKS"]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr", "-I", INCLUDE,
              "-I", CSRC]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfp4q.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def up_to_date(path: str = LIBPATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile and link; returns the library path."""
    libpath = DEBUG_LIBPATH if debug else LIBPATH
    if not force and up_to_date(libpath):
        return libpath
    nvcc = nvcc_path()
    objdir = os.path.join(LIBDIR, "obj_debug" if debug else "obj")
    os.makedirs(objdir, exist_ok=True)
    flags = [*extra_flags, *(DEBUG_FLAGS if debug else [])]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = libpath + ".tmp"
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, libpath)
    return libpath


if __name__ == "__main__":
    force = "--force" in sys.argv
    verbose = "--verbose" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    if extra:
        force = True
        verbose = True
    print(build(force=force, verbose=verbose, extra_flags=extra, debug="--debug" in sys.argv))
