"""Builds the sm_103a shared library in-tree with nvcc.

    python -m scaled_dot_product_08_gb300.build

Each translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into _lib/libsdpa08.so (CUDA runtime linked
statically, so the library needs only the NVIDIA driver at run time).

    python -m scaled_dot_product_08_gb300.build --debug

builds the same sources with -DATTN_DEBUG (in-kernel index checks) into
_lib/libsdpa08_debug.so, under _build_debug/.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libsdpa08.so")
DEBUG_LIB = os.path.join(LIBDIR, "libsdpa08_debug.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

SOURCES = ["attn_api.cu", "attn_fwd.cu", "attn_fwd_persist.cu", "attn_fwd_fp8.cu", "attn_bwd.cu", "attn_bwd_persist.cu", "attn_bwd_prep.cu", "attn_bwd_dq.cu",
           "attn_bwd_dq_persist.cu",
           "attn_decode.cu", "attn_mask.cu", "attn_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "attn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library; debug:
    the build with the in-kernel index checks (-DATTN_DEBUG)."""
    lib_path = DEBUG_LIB if debug else LIB
    if not force and up_to_date(lib_path):
        return lib_path
    build_dir = BUILD + "_debug" if debug else BUILD
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    extra = ["-DATTN_DEBUG"] if debug else []

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
