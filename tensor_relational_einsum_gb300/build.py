"""Build libea.so in-tree for sm_103a with nvcc (no cmake, no setuptools).

Every translation unit is compiled in parallel into ``_build/`` and linked
into ``tensor_relational_einsum_gb300/libea.so`` against the shared CUDA
runtime (the one PyTorch also loads).  A rebuild happens only when a source
or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libea.so")
# The bounds-checking build (EA_DEBUG_BOUNDS: every kernel checks each
# tile's element range against its arena before touching it).  The binding
# loads it instead of libea.so when the environment sets EA_BOUNDS_CHECK=1.
LIB_BOUNDS = os.path.join(PKG, "libea_bounds.so")


def bounds_variant() -> bool:
    return os.environ.get("EA_BOUNDS_CHECK", "") == "1"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libea.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(root, "lib64")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cpp")) + glob.glob(os.path.join(CSRC, "kernels", "*.cu")))


def headers():
    return (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "kernels", "*.cuh")) +
            [os.path.join(INCLUDE, "ea.h")])


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in sources() + headers() + [__file__])


def build(force: bool = False, verbose: bool = False, extra_flags=(), bounds: bool | None = None) -> str:
    """Build libea.so (or, with bounds=True -- by default when EA_BOUNDS_CHECK=1
    -- the bounds-checking libea_bounds.so) if a source is newer; return its path."""
    if bounds is None:
        bounds = bounds_variant()
    lib = LIB_BOUNDS if bounds else LIB
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, "bounds") if bounds else BUILD
    os.makedirs(objdir, exist_ok=True)
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *extra_flags,
              *(["-DEA_DEBUG_BOUNDS"] if bounds else [])]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.relpath(src, CSRC).replace(os.sep, "_") + ".o")
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-lineinfo", *common, "-c", src, "-o", obj]
        else:
            cmd = [nvcc, *ARCH, *common, "-x", "c++", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp.{os.getpid()}"
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-L", libdir, "-Xlinker",
           f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=(["-Xptxas", "-v"] if "--ptxas" in sys.argv else []),
                bounds=True if "--bounds" in sys.argv else None))
