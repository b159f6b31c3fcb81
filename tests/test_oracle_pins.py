"""Pins of the CPU oracle against facts that do not come from the oracle.

Rule being pinned: HyperQwen lookup-drafting article (kwkr.cn/news/564408),
section "第1步" -- longest current suffix of min_m..max_m tokens, its most recent
earlier occurrence (overlap with the suffix allowed), the following tokens as the
draft, read from the self-extended history e[L+j] = e[p+m+j].

  * hand-worked fixtures (tests/golden/hand_worked.txt);
  * planted verbatim copies, whose (m, p) and draft are known by construction;
  * the closed form of purely periodic histories (the overlap rule);
  * exhaustive enumeration of tiny histories over 2-4 letter alphabets, each
    result checked against the defining invariants (tests/invariants.py);
  * the invariants again on all five synthetic workloads;
  * special cases (empty batch, L in {0, 1, min_m, min_m+1}, K = 0, ...).
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest

import gen
import oracle
from goldens import load_cases
from invariants import check_batch, check_small

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c.name)
def test_hand_worked(case, lib):
    draft, length, pos, m = oracle.lookup_draft(case.tokens, case.offsets, case.min_m,
                                                case.max_m, case.K, lib=lib)
    np.testing.assert_array_equal(m, case.expect_m)
    np.testing.assert_array_equal(pos, case.expect_pos)
    np.testing.assert_array_equal(length, case.expect_len)
    np.testing.assert_array_equal(draft, case.expect_draft)


def test_planted_tiny(lib):
    """tiny: four requests end in a 64-token copy of t[s0 : s0+64].  The 12-suffix is
    t[s0+52 : s0+64], so m = 12, p = s0 + 52 and the draft is t[s0+64 : s0+79].
    The other four, uniform over 32000 tokens, have no 4-gram repeat of their suffix
    (chance about 4096 * 32000^-4), so they must report no match."""
    w = gen.make_workload("tiny")
    draft, length, pos, m = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, lib=lib)
    assert len(w.planted) == 4
    for r in range(w.B):
        t = w.tokens[w.offsets[r]:w.offsets[r + 1]]
        if r in w.planted:
            s0, c = w.planted[r]
            assert (m[r], pos[r], length[r]) == (12, s0 + c - 12, 15)
            np.testing.assert_array_equal(draft[r], t[s0 + c:s0 + c + 15])
        else:
            assert (m[r], pos[r], length[r]) == (0, -1, 0)
            assert np.all(draft[r] == -1)


@pytest.mark.parametrize("name", ["recitation25k", "ragged262k", "chats"])
def test_planted_copies(name, lib):
    """Requests that end c >= 12 tokens into a copy of t[s0 : s0+c] match at m = 12,
    p = s0 + c - 12 (a more recent chance 12-gram repeat of Zipf text has
    probability far below 1e-15), and draft t[s0+c : s0+c+K]."""
    w = gen.make_workload(name)
    draft, length, pos, m = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K,
                                                threads=4, lib=lib)
    checked = 0
    for r, (s0, c) in w.planted.items():
        if c < w.max_m:
            continue
        t = w.tokens[w.offsets[r]:w.offsets[r + 1]]
        assert (m[r], pos[r], length[r]) == (12, s0 + c - 12, w.K), r
        np.testing.assert_array_equal(draft[r], t[s0 + c:s0 + c + w.K])
        checked += 1
    assert checked >= len(w.planted) * 0.9


@pytest.mark.parametrize("d", list(range(1, 16)) + [29, 40])
@pytest.mark.parametrize("L_extra", [0, 1, 5, 37])
def test_periodic_closed_form(d, L_extra, lib):
    """t[i] = a[i mod d] with d distinct tokens and L >= d + max_m: every length up to
    max_m matches, the latest earlier start of the max_m-suffix is one period back,
    p = L - max_m - d (overlapping the suffix when d < max_m), and the draft
    continues the period, draft[j] = a[(L + j) mod d]."""
    max_m, min_m, K = 12, 4, 15
    rng = np.random.default_rng(d * 100 + L_extra)
    a = rng.permutation(1000)[:d].astype(np.int32) - 300
    L = d + max_m + L_extra
    t = a[np.arange(L) % d]
    offsets = np.array([0, L], dtype=np.int64)
    draft, length, pos, m = oracle.lookup_draft(t, offsets, min_m, max_m, K, lib=lib)
    assert (m[0], pos[0], length[0]) == (max_m, L - max_m - d, K)
    np.testing.assert_array_equal(draft[0], a[(L + np.arange(K)) % d])


def test_periodic_short_history(lib):
    """A history of one period plus a partial one, L < d + max_m: the suffix of length
    L - d (< max_m) is the longest with an earlier occurrence, at p = 0."""
    a = np.arange(10, 17, dtype=np.int32)          # d = 7 distinct tokens
    t = np.concatenate([a, a[:5]])                   # L = 12, max admissible m = 5
    offsets = np.array([0, t.size], dtype=np.int64)
    draft, length, pos, m = oracle.lookup_draft(t, offsets, 2, 12, 4, lib=lib)
    assert (m[0], pos[0]) == (5, 0)
    np.testing.assert_array_equal(draft[0], a[[5, 6, 0, 1]])


def _all_histories(alphabet: int, max_len: int):
    for L in range(0, max_len + 1):
        for seq in itertools.product(range(alphabet), repeat=L):
            yield list(seq)


@pytest.mark.parametrize("alphabet,max_len", [(2, 12), (3, 8), (4, 6)])
@pytest.mark.parametrize("min_m,max_m,K", [(1, 3, 5), (2, 4, 1), (4, 12, 5), (2, 2, 3), (1, 1, 2)])
def test_exhaustive_invariants(alphabet, max_len, min_m, max_m, K, lib):
    """Every history over a tiny alphabet up to a length: the oracle's answer must
    satisfy the defining invariants, which fix it uniquely."""
    hists = list(_all_histories(alphabet, max_len))
    lengths = [len(h) for h in hists]
    tokens = np.array([x for h in hists for x in h], dtype=np.int32)
    offsets = gen.offsets_from_lengths(lengths)
    draft, length, pos, m = oracle.lookup_draft(tokens, offsets, min_m, max_m, K, lib=lib)
    bad = []
    for r, h in enumerate(hists):
        msg = check_small(h, min_m, max_m, K, int(m[r]), int(pos[r]), int(length[r]), draft[r])
        if msg:
            bad.append((h, msg))
            if len(bad) > 5:
                break
    assert not bad, bad


@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_invariants_on_workloads(name, lib):
    w = gen.make_workload(name)
    draft, length, pos, m = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K,
                                                threads=4, lib=lib)
    errors = check_batch(w.tokens, w.offsets, w.min_m, w.max_m, w.K, m, pos, length, draft)
    assert not errors, errors[:5]


def test_special_cases(lib):
    # empty batch
    d, ln, p, m = oracle.lookup_draft(np.zeros(0, np.int32), np.zeros(1, np.int64), 4, 12, 15, lib=lib)
    assert d.shape == (0, 15) and ln.size == 0
    # L in {0, 1, min_m, min_m + 1}, all tokens equal: only L = min_m + 1 can match
    min_m, max_m, K = 4, 12, 3
    lengths = [0, 1, min_m, min_m + 1]
    tokens = np.full(sum(lengths), 9, dtype=np.int32)
    d, ln, p, m = oracle.lookup_draft(tokens, gen.offsets_from_lengths(lengths),
                                      min_m, max_m, K, lib=lib)
    np.testing.assert_array_equal(m, [0, 0, 0, min_m])
    np.testing.assert_array_equal(p, [-1, -1, -1, 0])
    np.testing.assert_array_equal(ln, [0, 0, 0, K])
    np.testing.assert_array_equal(d[3], [9, 9, 9])
    # arguments that describe no valid step are rejected
    one = np.ones(4, np.int32)
    offs = np.array([0, 4], np.int64)
    for bad in [(0, 4, 1), (5, 4, 1), (2, 4, -1)]:
        with pytest.raises(ValueError):
            oracle.lookup_draft(one, offs, *bad, lib=lib)


def test_cross_request_boundary(lib):
    """The previous request's tail equals the next request's suffix: the match must
    not leave the request (and here the request alone has no match)."""
    rng = np.random.default_rng(7)
    a = rng.integers(0, 1 << 20, size=3000).astype(np.int32)
    b = rng.integers(0, 1 << 20, size=3000).astype(np.int32)
    b[-12:] = a[-12:]
    tokens = np.concatenate([a, b])
    offsets = np.array([0, a.size, a.size + b.size], dtype=np.int64)
    d, ln, p, m = oracle.lookup_draft(tokens, offsets, 4, 12, 5, lib=lib)
    assert (m[1], p[1], ln[1]) == (0, -1, 0)


def test_threaded_equals_serial(lib):
    w = gen.make_workload("chats")
    a = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=1, lib=lib)
    b = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=6, lib=lib)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
