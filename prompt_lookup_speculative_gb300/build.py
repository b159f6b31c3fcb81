"""Compile the CUDA library in-tree for GB300 (sm_103a).

The library is five translation units, ``csrc/lookup_draft.cu`` (the drafting
step), ``csrc/lookup_loop.cu`` (the decode-loop steps around it),
``csrc/lookup_index.cu`` (the incremental n-gram index),
``csrc/lookup_ctxcache.cu`` (context-cache drafting) and ``csrc/read_floor.cu``
(a measurement aid: a plain streaming read), built with nvcc into
``_build/liblookup_draft.so`` next to this file.  The drafting step's source is
also compiled with LOOKUP_DRAFT_CHECKED=1 into ``_build/liblookup_draft_checked.so``:
the same entry points with device-side index checks (include/lookup_draft.h).  The CUDA runtime is linked
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
# The checked build of the drafting step (LOOKUP_DRAFT_CHECKED=1; read_floor.cu rides along
# so that it exports everything lookup_draft.h declares): device-side
# index checks that set bits in a check word instead of faulting.
CHECKED_SOURCES = [os.path.join(PKG_DIR, "csrc", f) for f in ("lookup_draft.cu", "read_floor.cu")]
CHECKED_LIB_PATH = os.path.join(BUILD_DIR, "liblookup_draft_checked.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def compile_command(out: str, extra: list[str] | None = None, checked: bool = False) -> list[str]:
    """nvcc command line of the library (checked=True: the checked build of the
    drafting step)."""
    sources = CHECKED_SOURCES if checked else SOURCES
    defines = ["-DLOOKUP_DRAFT_CHECKED=1"] if checked else []
    return [nvcc_path(), *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17",
            "-Xcompiler", "-fPIC,-O2", "-shared", "-cudart", "static",
            "-I", INCLUDE_DIR, *defines, "-o", out, *sources, *(extra or [])]


def up_to_date() -> bool:
    for lib in (LIB_PATH, CHECKED_LIB_PATH):
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if not all(os.path.getmtime(p) <= t for p in SOURCES + HEADERS + [__file__]):
            return False
    return True


def build(force: bool = False, verbose: bool = False) -> str:
    """Build both libraries (regular and checked, compiled side by side) if either
    is missing or stale; return the regular library's path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else None
    jobs = []
    for lib, checked in ((LIB_PATH, False), (CHECKED_LIB_PATH, True)):
        tmp = lib + f".tmp{os.getpid()}"
        jobs.append((subprocess.Popen(compile_command(tmp, extra, checked)), tmp, lib))
    failed = [p.args for p, _, _ in jobs if p.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    for _, tmp, lib in jobs:
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
