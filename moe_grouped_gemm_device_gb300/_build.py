"""Compile the CUDA sources of the package into an in-tree shared library.

``build()`` runs nvcc once per translation unit (in parallel) for sm_103a
only, then links ``_build/librg.so`` with the CUDA runtime linked statically,
so loading the library needs no GPU and no libcudart on the search path.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "librg.so")
SOURCES = ["api.cu", "mgemm.cu", "kgemm.cu", "mxgemm.cu", "selftest.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("ptx.cuh", "internal.h", "bounds.cuh", "kgemm_plan.cuh")] + [os.path.join(INCLUDE, "rg.h")]
# The debug-bounds build: every copy and store coordinate the kernels compute
# is checked against its operand; a failed check sets RG_DEV_BOUNDS and the
# access is skipped.  Built on request into its own directory.
BOUNDS_DIR = os.path.join(OUT_DIR, "bounds")
BOUNDS_FLAGS = ("-DRG_DEBUG_BOUNDS=1",)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librg.so")


def _inputs():
    return [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [__file__]


def is_stale(lib: str = None) -> bool:
    lib = lib or LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_dir: str = None) -> str:
    """Build librg.so into out_dir (default: the package's _build directory)
    with extra nvcc flags; returns the library's path."""
    out_dir = out_dir or OUT_DIR
    lib = os.path.join(out_dir, "librg.so")
    if not force and not is_stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_bounds(force: bool = False) -> str:
    """The debug-bounds build of the library (see BOUNDS_FLAGS)."""
    return build(force=force, extra_flags=BOUNDS_FLAGS, out_dir=BOUNDS_DIR)


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, extra_flags=sys.argv[1:]))
