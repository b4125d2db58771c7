"""Build libxs_paged.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the shared library links the
CUDA runtime dynamically so it shares the process's runtime (and current
device) with PyTorch.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libxs_paged.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
# The debug library: the same sources compiled with -DXS_DEBUG_BOUNDS, so every
# computed global-memory index is checked in the kernels (XS_FLAG_BOUNDS).
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_BUILD_DIR, "libxs_paged_debug.so")
SOURCES = ["kv_append.cu", "paged_decode.cu", "kv_swap.cu", "block_alloc.cu", "paged_prefill_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libxs_paged")
    return cand


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "xs_paged.h"))
    return files


def up_to_date(debug_bounds: bool = False) -> bool:
    lib = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug_bounds: bool = False) -> str:
    """Build the release library (or, with debug_bounds, the debug library with
    in-kernel bounds checks) unless it is newer than every source; returns its path."""
    build_dir = DEBUG_BUILD_DIR if debug_bounds else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    if not force and up_to_date(debug_bounds):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    flags = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
             "-I", CSRC, *(["-DXS_DEBUG_BOUNDS"] if debug_bounds else []), *(extra_flags or [])]
    if verbose:
        flags += ["-Xptxas", "-v"]
    exe = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [exe, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
