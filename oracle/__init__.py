"""CPU oracle for prompt-lookup drafting -- TEST INFRASTRUCTURE ONLY.

The oracle is plain C in this directory, compiled with gcc and called through
ctypes:
  lookup_oracle.c  one batched draft step, brute force (HyperQwen lookup-drafting
                   article, section "第1步": longest current suffix of min_m..max_m
                   tokens, its most recent earlier occurrence, overlap with the
                   suffix allowed, the following tokens as the draft);
  loop_oracle.c    the decode-loop steps around it ("第2步", "第3步");
  ctx_oracle.c     context-cache drafting (llama.cpp prompt-lookup article);
  policy_oracle.c  the draft-source controller (Strata engine article, section 五).

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
_SRCS = [os.path.join(_HERE, f) for f in ("lookup_oracle.c", "loop_oracle.c", "ctx_oracle.c", "policy_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblookup_oracle.so")

_lib = None
_lock = threading.Lock()
_pools: dict[int, ThreadPoolExecutor] = {}


def _pool(threads: int) -> ThreadPoolExecutor:
    """A thread pool of `threads` workers kept for the life of the process (making
    one per call cost milliseconds, more than a whole batch on many cores)."""
    with _lock:
        ex = _pools.get(threads)
        if ex is None:
            ex = _pools[threads] = ThreadPoolExecutor(max_workers=threads)
        return ex


def build(force: bool = False) -> str:
    """Compile the oracle into a shared object next to its source; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wextra",
                    "-o", tmp, *_SRCS], check=True)
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
    vp = ctypes.c_void_p
    lib.oracle_fuse.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.oracle_fuse.restype = ctypes.c_int
    lib.oracle_schedule.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.oracle_schedule.restype = ctypes.c_int
    lib.oracle_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp]
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_append.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp]
    lib.oracle_append.restype = ctypes.c_int
    if hasattr(lib, "oracle_ctx_draft"):
        lib.oracle_ctx_draft.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        lib.oracle_ctx_draft.restype = ctypes.c_int
    if hasattr(lib, "oracle_policy"):
        f32 = ctypes.c_float
        lib.oracle_policy.argtypes = [vp, vp, i32, i32, i32, f32, f32, f32, f32, f32, i32, i32, i32, vp, vp, vp]
        lib.oracle_policy.restype = ctypes.c_int
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
    # Balance by history length: cut the request range at equal token counts, one
    # piece per thread (each piece is one C call; many short calls queue on the
    # interpreter lock as they return).
    work = (offsets[1:] - offsets[:-1]).astype(np.float64) + 64.0
    cum = np.concatenate([[0.0], np.cumsum(work)])
    pieces = min(B, threads)
    cuts = np.searchsorted(cum, np.linspace(0.0, cum[-1], pieces + 1), side="left")
    cuts[0], cuts[-1] = 0, B
    cuts = np.unique(np.clip(cuts, 0, B))
    rcs = list(_pool(threads).map(lambda ab: run(int(ab[0]), int(ab[1])), zip(cuts[:-1], cuts[1:])))
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


# ------------------------------------------------------------- loop steps ----
def _arr(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


def fuse(lookup_draft, lookup_mlen, model_draft, long_block, H: int, T: int, replace_min: int = 8,
         agree_min: int = 6, agree_n: int = 2, tail_min: int = 4, lib=None):
    """Fusion of lookup drafts with draft-model proposals (HyperQwen article, "第2步").
    Returns (block [B][H+T], len [B], point_mass [B][H+T])."""
    lib = lib or load()
    ld = _arr(lookup_draft, np.int32)
    lm = _arr(lookup_mlen, np.int32)
    md = _arr(model_draft, np.int32)
    lg = _arr(long_block, np.int32)
    B, K = ld.shape
    block = np.empty((B, H + T), np.int32)
    ln = np.empty(B, np.int32)
    pm = np.empty((B, H + T), np.int32)
    rc = lib.oracle_fuse(_p(ld), _p(lm), _p(md), _p(lg), B, K, H, T, replace_min, agree_min, agree_n,
                         tail_min, _p(block), _p(ln), _p(pm))
    if rc:
        raise ValueError("oracle_fuse rejected the arguments")
    return block, ln, pm


def schedule(lookup_mlen, committed, state, H: int, T: int, tail_min: int = 4, slack: int = 1,
             enter_steps: int = 2, sticky: int = 3, lib=None):
    """One long-block scheduling update ("第3步"); `state` [B][3] is updated in place.
    Returns out_long [B]."""
    lib = lib or load()
    lm = _arr(lookup_mlen, np.int32)
    cm = _arr(committed, np.int32)
    assert state.dtype == np.int32 and state.flags["C_CONTIGUOUS"]
    B = lm.shape[0]
    out = np.empty(B, np.int32)
    rc = lib.oracle_schedule(_p(lm), _p(cm), B, H, T, tail_min, slack, enter_steps, sticky,
                             _p(state), _p(out))
    if rc:
        raise ValueError("oracle_schedule rejected the arguments")
    return out


def policy(lookup_mlen, accepted, acc, prev, n_lookup: int, n_model: int, t_lookup: float, t_model: float,
           t_plain: float, alpha: float = 0.125, margin: float = 0.05, edges=(6, 8, 12), lib=None):
    """One step of the draft-source controller (Strata engine article, section 五);
    ``acc`` float32 [B][5] and ``prev`` int32 [B][3] are updated in place.  Returns
    the choice per request: 0 plain decoding, 1 the draft model, 2 the lookup draft."""
    lib = lib or load()
    lm = _arr(lookup_mlen, np.int32)
    ac = _arr(accepted, np.int32)
    assert acc.dtype == np.float32 and acc.flags["C_CONTIGUOUS"] and acc.shape == (lm.shape[0], 5)
    assert prev.dtype == np.int32 and prev.flags["C_CONTIGUOUS"] and prev.shape == (lm.shape[0], 3)
    B = lm.shape[0]
    out = np.empty(B, np.int32)
    rc = lib.oracle_policy(_p(lm), _p(ac), B, n_lookup, n_model, t_lookup, t_model, t_plain, alpha, margin,
                           int(edges[0]), int(edges[1]), int(edges[2]), _p(acc), _p(prev), _p(out))
    if rc:
        raise ValueError("oracle_policy rejected the arguments")
    return out


def verify(block, length, target, probs=None, qprobs=None, point_mass=None, u=None, lib=None):
    """Greedy (probs None) or sampled verification of proposal blocks.
    Returns (accepted [B], commit [B][P+1], ncommit [B])."""
    lib = lib or load()
    bl = _arr(block, np.int32)
    ln = _arr(length, np.int32)
    tg = _arr(target, np.int32)
    pr, qp, pm, uu = _arr(probs, np.float32), _arr(qprobs, np.float32), _arr(point_mass, np.int32), _arr(u, np.float32)
    B, P = bl.shape
    acc = np.empty(B, np.int32)
    commit = np.empty((B, P + 1), np.int32)
    nc = np.empty(B, np.int32)
    rc = lib.oracle_verify(_p(bl), _p(ln), _p(tg), _p(pr), _p(qp), _p(pm), _p(uu), B, P,
                           _p(acc), _p(commit), _p(nc))
    if rc:
        raise ValueError("oracle_verify rejected the arguments")
    return acc, commit, nc


def append(tokens, offsets, commit, ncommit, lib=None):
    """The next CSR batch: every history followed by its committed tokens."""
    lib = lib or load()
    tk = _arr(tokens, np.int32)
    of = _arr(offsets, np.int64)
    cm = _arr(commit, np.int32)
    nc = _arr(ncommit, np.int32)
    B, W = cm.shape
    total = int(of[-1] - of[0]) + int(nc.sum())
    out_t = np.empty(total, np.int32)
    out_o = np.empty(B + 1, np.int64)
    rc = lib.oracle_append(_p(tk), _p(of), _p(cm), _p(nc), B, W, _p(out_t), _p(out_o))
    if rc:
        raise ValueError("oracle_append rejected the arguments")
    return out_t, out_o


# ----------------------------------------------------------- context cache ----
def ctx_draft(tokens, offsets, K: int, n_min: int = 1, n_max: int = 4, min_count=(1, 1, 1, 1),
              share=((1, 2), (1, 2), (1, 2), (1, 2)), threads: int = 1, lib=None):
    """Context-cache drafting (llama.cpp prompt-lookup article): for each request,
    up to K tokens, each the most frequent next token of the longest n-gram
    (n_max .. n_min) of the context that passes the thresholds (count >=
    min_count[n-1], share of the top next token >= share[n-1] = (num, den)).
    Returns (draft [B, K] int32 (-1 past the end), len [B] int32)."""
    lib = lib or load()
    tk = np.ascontiguousarray(tokens, dtype=np.int32)
    of = np.ascontiguousarray(offsets, dtype=np.int64)
    B = int(of.shape[0]) - 1
    mc = np.ascontiguousarray(min_count, dtype=np.int32)
    num = np.ascontiguousarray([s[0] for s in share], dtype=np.int32)
    den = np.ascontiguousarray([s[1] for s in share], dtype=np.int32)
    draft = np.empty((max(B, 0), K), np.int32)
    length = np.empty(max(B, 0), np.int32)
    if B <= 0:
        return draft, length

    def run(lo, hi):
        return lib.oracle_ctx_draft(_p(tk), _p(of), lo, hi, n_min, n_max, K, _p(mc), _p(num), _p(den),
                                    _p(draft), _p(length))

    if threads <= 1 or B == 1:
        rcs = [run(0, B)]
    else:
        cuts = np.linspace(0, B, min(B, threads) + 1).astype(int)
        rcs = list(_pool(threads).map(lambda ab: run(int(ab[0]), int(ab[1])), zip(cuts[:-1], cuts[1:])))
    if any(rcs):
        raise ValueError("oracle_ctx_draft rejected the arguments")
    return draft, length
