"""Defining properties of one drafting result, checked without searching for it.

For a history t[0..L) and a reported match (m, p) (m = 0: no match), the result
of the longest-then-most-recent rule (HyperQwen lookup-drafting article,
section "第1步") is the unique one for which all of these hold:

  (i)   found:    min_m <= m <= max_m, 0 <= p, p + m <= L - 1, and
                  t[p:p+m] == t[L-m:L]  (the occurrence is earlier than the
                  suffix itself but may overlap it);
  (ii)  longest:  the suffix one token longer (or, with no match, the min_m
                  suffix) occurs at no admissible start, when that length is
                  <= min(max_m, L-1).  An occurrence longer by more than one
                  contains one longer by exactly one, so one length suffices;
  (iii) latest:   no start p' in (p, L-m-1] matches at length m;
  (iv)  draft:    with d = L - p - m, draft[j] = t[p + m + (j mod d)], which is
                  the closed form of the self-extended history e[L+j] = e[p+m+j];
                  a match yields length K and position p, no match yields
                  length 0, position -1 and -1 in every draft slot.

These are checks of a result, not a second search, so they pin an
implementation independently of how it searches.
"""
from __future__ import annotations

import numpy as np


def _occurs_list(t: list, L: int, n: int, lo: int, hi: int) -> bool:
    """Some start p in [lo, hi] with t[p:p+n] == t[L-n:L] (list version)."""
    suf = t[L - n:L]
    for p in range(max(lo, 0), min(hi, L - n - 1) + 1):
        if t[p:p + n] == suf:
            return True
    return False


def check_small(t: list, min_m: int, max_m: int, K: int,
                m: int, pos: int, length: int, draft) -> str | None:
    """Check one result on a short Python-list history; return a message or None."""
    L = len(t)
    draft = list(draft)
    if m == 0:
        if length != 0 or pos != -1 or any(x != -1 for x in draft):
            return f"no-match sentinels wrong: len={length} pos={pos} draft={draft}"
        if min_m <= min(max_m, L - 1) and _occurs_list(t, L, min_m, 0, L):
            return f"reported no match but the {min_m}-suffix occurs earlier"
        return None
    p = pos
    if not (min_m <= m <= max_m and p >= 0 and p + m <= L - 1):
        return f"(m={m}, p={p}) outside the admissible range for L={L}"
    if t[p:p + m] != t[L - m:L]:
        return f"(m={m}, p={p}) is not an occurrence of the suffix"
    if m + 1 <= min(max_m, L - 1) and _occurs_list(t, L, m + 1, 0, L):
        return f"a longer ({m + 1}) occurrence exists"
    if _occurs_list(t, L, m, p + 1, L):
        return f"a later occurrence of length {m} exists"
    d = L - p - m
    want = [t[p + m + (j % d)] for j in range(K)]
    if length != K or draft != want:
        return f"draft wrong: len={length} draft={draft} want={want}"
    return None


def occurrences(t: np.ndarray, n: int) -> np.ndarray:
    """Boolean over starts p in [0, L-n-1]: t[p:p+n] == t[L-n:L]."""
    L = t.shape[0]
    count = L - n
    if count <= 0:
        return np.zeros(0, dtype=bool)
    eq = np.ones(count, dtype=bool)
    for i in range(n):
        eq &= t[i:i + count] == t[L - n + i]
    return eq


def check_array(t: np.ndarray, min_m: int, max_m: int, K: int,
                m: int, pos: int, length: int, draft: np.ndarray) -> str | None:
    """Same checks as check_small, vectorised for long numpy histories."""
    L = int(t.shape[0])
    draft = np.asarray(draft)
    if m == 0:
        if length != 0 or pos != -1 or np.any(draft != -1):
            return f"no-match sentinels wrong: len={length} pos={pos}"
        if min_m <= min(max_m, L - 1) and occurrences(t, min_m).any():
            return f"reported no match but the {min_m}-suffix occurs earlier"
        return None
    p = pos
    if not (min_m <= m <= max_m and p >= 0 and p + m <= L - 1):
        return f"(m={m}, p={p}) outside the admissible range for L={L}"
    if not np.array_equal(t[p:p + m], t[L - m:L]):
        return f"(m={m}, p={p}) is not an occurrence of the suffix"
    if m + 1 <= min(max_m, L - 1) and occurrences(t, m + 1).any():
        return f"a longer ({m + 1}) occurrence exists"
    if occurrences(t, m)[p + 1:].any():
        return f"a later occurrence of length {m} exists"
    d = L - p - m
    want = t[p + m + (np.arange(K) % d)]
    if length != K or not np.array_equal(draft, want):
        return "draft differs from the closed form"
    return None


def check_batch(tokens: np.ndarray, offsets: np.ndarray, min_m: int, max_m: int, K: int,
                m, pos, length, draft) -> list[str]:
    errors = []
    for r in range(offsets.shape[0] - 1):
        t = tokens[offsets[r]:offsets[r + 1]]
        msg = check_array(t, min_m, max_m, K, int(m[r]), int(pos[r]), int(length[r]), draft[r])
        if msg:
            errors.append(f"request {r}: {msg}")
    return errors
