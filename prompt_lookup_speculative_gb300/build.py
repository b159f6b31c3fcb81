"""Compile the CUDA library in-tree for GB300 (sm_103a).

The library is five translation units, ``csrc/lookup_draft.cu`` (the drafting
step), ``csrc/lookup_loop.cu`` (the decode-loop steps around it),
``csrc/lookup_index.cu`` (the incremental n-gram index),
``csrc/lookup_ctxcache.cu`` (context-cache drafting) and ``csrc/read_floor.cu``
(a measurement aid: a plain streaming read), built with nvcc into
``_build/liblookup_draft.so`` next to this file.  The CUDA runtime is linked
statically, so the library loads on a machine without a GPU (its calls then
fail with a CUDA error) and needs nothing from the Python environment.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
INCLUDE_DIR = os.path.join(REPO_DIR, "include")
SOURCES = [os.path.join(PKG_DIR, "csrc", f)
           for f in ("lookup_draft.cu", "lookup_loop.cu", "lookup_index.cu", "lookup_ctxcache.cu",
                     "read_floor.cu")]
HEADERS = [os.path.join(INCLUDE_DIR, f)
           for f in ("lookup_draft.h", "lookup_loop.h", "lookup_index.h", "lookup_ctxcache.h")] + \
          [os.path.join(PKG_DIR, "csrc", "common.cuh")]
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liblookup_draft.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def compile_command(out: str, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17",
            "-Xcompiler", "-fPIC,-O2", "-shared", "-cudart", "static",
            "-I", INCLUDE_DIR, "-o", out, *SOURCES, *(extra or [])]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in SOURCES + HEADERS + [__file__])


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the library if it is missing or stale; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = compile_command(tmp, ["-Xptxas", "-v"] if verbose else None)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
