"""Build libpkv.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
``paged_kv_cache_234_gb300/_build/libpkv.so`` with the CUDA runtime linked
statically, so the library depends only on the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libpkv.so")
DEBUG_LIB_PATH = os.path.join(BUILD_DIR, "libpkv_debug.so")
INCLUDE = os.path.join(os.path.dirname(PKG_DIR), "include")
SOURCES = ("pkv_host.cu", "pkv_quantize.cu", "pkv_decode.cu", "pkv_append.cu", "pkv_evict.cu",
           "pkv_copy.cu", "pkv_block_manager.cpp")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pkv.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


DEBUG_SOURCES = ("pkv_decode.cu", "pkv_evict.cu")  # the kernels with PKV_DEBUG checks


def build_debug() -> str:
    """libpkv_debug.so: the library with the decode and eviction kernels built
    with PKV_DEBUG (shared-memory address and index checks, read back by
    pkv_debug_flags / pkv_debug_evict_flags).  For tests; the release library
    is untouched."""
    build()
    if os.path.exists(DEBUG_LIB_PATH) and all(
            os.path.getmtime(f) <= os.path.getmtime(DEBUG_LIB_PATH) for f in _inputs()):
        return DEBUG_LIB_PATH
    nvcc = _nvcc()

    def compile_debug(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + "_debug.o")
        cmd = [nvcc] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                               "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-DPKV_DEBUG",
                               "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for the debug {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with concurrent.futures.ThreadPoolExecutor(len(DEBUG_SOURCES)) as ex:
        dbg = list(ex.map(compile_debug, DEBUG_SOURCES))
    objs = [os.path.join(BUILD_DIR, os.path.splitext(f)[0] + ".o") for f in SOURCES
            if f not in DEBUG_SOURCES] + dbg
    tmp = DEBUG_LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, DEBUG_LIB_PATH)
    return DEBUG_LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
