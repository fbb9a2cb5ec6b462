"""Build the in-tree CUDA library ``_lib/libsgemm_gb300.so`` for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically (the driver API is reached
through ``cudaGetDriverEntryPointByVersion``, so no ``-lcuda``).
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libsgemm_gb300.so")
OBJ_DIR = os.path.join(ROOT, "_build", "obj")
# Debug build: the same sources with the kernels' device-side index checks compiled
# in (SGEMM_DEBUG_CHECKS=1; a failed check records SGEMM_ERR_INDEX and skips its
# access). The binding loads it when SGEMM_GB300_DEBUG_CHECKS=1.
DEBUG_LIB = os.path.join(OUT_DIR, "libsgemm_gb300_debug.so")
DEBUG_OBJ_DIR = os.path.join(ROOT, "_build", "obj_debug")

SOURCES = ["ffma_kernels.cu", "tf32_kernels.cu", "min2_kernels.cu", "ladder_kernels.cu", "planner.cpp", "sgemm_api.cpp", "static_scratch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return path


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}"] + list(extra)


def _deps():
    """Newest modification time of everything the library is built from."""
    inc = os.path.join(ROOT, "include")
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h", ".cpp"))]
    files += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    """Compile and link the library (or, with `debug`, its index-checking variant) if
    any source is newer than it; return its path."""
    lib_path = DEBUG_LIB if debug else LIB
    obj_dir = DEBUG_OBJ_DIR if debug else OBJ_DIR
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _deps():
        return lib_path
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DSGEMM_DEBUG_CHECKS=1"] if debug else [])

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + _flags(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
