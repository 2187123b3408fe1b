"""Compile the CUDA library (libmkv.so) in-tree for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then
nvcc links the shared library. The CUDA runtime is linked statically, so the
library needs nothing on LD_LIBRARY_PATH. Usage: ``python -m
geometric_kv_cache_gb300.build`` or ``build_library()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
OUT_DIR = os.path.join(PKG_DIR, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "libmkv.so")
SOURCES = ["mkv_kernels.cu", "mkv_gather.cu", "mkv_inplace.cu", "mkv_summaries.cu", "mkv_oja.cu", "mkv_piece.cu", "mkv_api.cu", "mkv_noalloc.cu"]
HEADERS = [os.path.join(CSRC, "mkv_internal.h"), os.path.join(CSRC, "mkv_device.cuh"),
           os.path.join(CSRC, "mkv_select.cuh"), os.path.join(CSRC, "mkv_gather.cuh"),
           os.path.join(os.path.dirname(PKG_DIR), "include", "mkv.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-ffp-contract=off",
                           "--fmad=true"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmkv.so")


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Build libmkv.so if missing or older than its sources; return its path."""
    if not force and not _stale():
        return LIB_PATH
    nvcc = nvcc_path()
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out, file=sys.stderr)
        if p.returncode != 0:
            failed.append((cmd, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + " ".join(link) + "\n" + r.stdout)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True,
                        extra_flags=("-Xptxas", "-v") if "--ptxas-v" in sys.argv else ()))
