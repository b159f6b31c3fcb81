"""CPU oracle for prompt-lookup drafting -- TEST INFRASTRUCTURE ONLY.

The oracle is ``lookup_oracle.c`` in this directory: a plain brute-force
statement of one batched draft step (HyperQwen lookup-drafting article,
section "第1步": longest current suffix of min_m..max_m tokens, its most recent
earlier occurrence, overlap with the suffix allowed, the following tokens as
the draft).  This module compiles it with gcc and calls it through ctypes.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library never does, and
the two share no code.

Every function of the oracle is pinned by ``-m "not gpu"`` tests against values
that do not come from the oracle itself: hand-worked fixtures, planted verbatim
copies with known answers, the closed form of periodic histories, exhaustive
enumeration on tiny alphabets checked against the defining invariants, and
special cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lookup_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblookup_oracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into a shared object next to its source; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wextra",
                    "-o", tmp, _SRC], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library, or a given build of it."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    p32 = ctypes.POINTER(ctypes.c_int32)
    p64 = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_lookup_draft.argtypes = [p32, p64, i32, i32, i32, i32, i32, p32, p32, p32, p32]
    lib.oracle_lookup_draft.restype = ctypes.c_int
    lib.oracle_find_match.argtypes = [p32, i64, i32, i32, p32, p64]
    lib.oracle_find_match.restype = ctypes.c_int
    lib.oracle_fill_draft.argtypes = [p32, i64, i32, i64, i32, p32]
    lib.oracle_fill_draft.restype = None
    return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def lookup_draft(tokens, offsets, min_m: int, max_m: int, K: int,
                 threads: int = 1, lib: ctypes.CDLL | None = None):
    """Run the oracle on a CSR batch held in host memory.

    tokens: int32 array; offsets: int64 array of B+1 entries.  Returns
    (draft[B, K] int32, length[B] int32, pos[B] int32, m[B] int32), where m is
    the match length (0 when there is no match).  With threads > 1 the requests
    are split into contiguous ranges run concurrently (ctypes drops the GIL).
    """
    lib = lib or load()
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    B = int(offsets.shape[0]) - 1
    draft = np.empty((max(B, 0), K), dtype=np.int32)
    length = np.empty(max(B, 0), dtype=np.int32)
    pos = np.empty(max(B, 0), dtype=np.int32)
    mlen = np.empty(max(B, 0), dtype=np.int32)
    if B <= 0:
        return draft, length, pos, mlen
    tp, op = _ptr(tokens, ctypes.c_int32), _ptr(offsets, ctypes.c_int64)
    dp, lp = _ptr(draft, ctypes.c_int32), _ptr(length, ctypes.c_int32)
    pp, mp = _ptr(pos, ctypes.c_int32), _ptr(mlen, ctypes.c_int32)

    def run(lo: int, hi: int) -> int:
        return lib.oracle_lookup_draft(tp, op, lo, hi, min_m, max_m, K, dp, lp, pp, mp)

    if threads <= 1 or B == 1:
        rc = run(0, B)
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return draft, length, pos, mlen
    # Balance by history length: cut the request range at equal token counts.
    work = (offsets[1:] - offsets[:-1]).astype(np.float64) + 64.0
    cum = np.concatenate([[0.0], np.cumsum(work)])
    pieces = min(B, threads * 8)
    cuts = np.searchsorted(cum, np.linspace(0.0, cum[-1], pieces + 1), side="left")
    cuts[0], cuts[-1] = 0, B
    cuts = np.unique(np.clip(cuts, 0, B))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        rcs = list(ex.map(lambda ab: run(int(ab[0]), int(ab[1])), zip(cuts[:-1], cuts[1:])))
    if any(rc != 0 for rc in rcs):
        raise ValueError("oracle rejected the arguments")
    return draft, length, pos, mlen


def find_match(history, min_m: int, max_m: int, lib: ctypes.CDLL | None = None):
    """(m, p) of the longest-then-latest earlier suffix occurrence, or (0, -1)."""
    lib = lib or load()
    t = np.ascontiguousarray(history, dtype=np.int32)
    m = ctypes.c_int32(0)
    p = ctypes.c_int64(-1)
    found = lib.oracle_find_match(_ptr(t, ctypes.c_int32), int(t.shape[0]), min_m, max_m,
                                  ctypes.byref(m), ctypes.byref(p))
    return (int(m.value), int(p.value)) if found else (0, -1)


def fill_draft(history, m: int, p: int, K: int, lib: ctypes.CDLL | None = None):
    """The K-token draft e[L..L+K) for a match (m, p) of the history."""
    lib = lib or load()
    t = np.ascontiguousarray(history, dtype=np.int32)
    out = np.empty(K, dtype=np.int32)
    lib.oracle_fill_draft(_ptr(t, ctypes.c_int32), int(t.shape[0]), m, p, K,
                          _ptr(out, ctypes.c_int32))
    return out
