"""Pins of the context-cache oracle (oracle/ctx_oracle.c) against hand-worked cases.

Rule (llama.cpp prompt-lookup article, section "Prompt lookup decoding 到底是什麼"):
n-grams of sizes 1..4 of the current stream; a draft token comes from an n-gram
that occurred before (count >= min_count) and whose most frequent next token
follows it at least half the time.  Readings: longest n first, one token at a
time with the drafted tokens extending the looked-up context, counts from the
history only, ties to the smallest token id.  Every expected value below is
worked out by hand in the comments, not taken from an implementation.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle


def draft1(hist, K, **kw):
    t = np.array(hist, np.int32)
    d, n = oracle.ctx_draft(t, np.array([0, len(t)], np.int64), K, **kw)
    return list(d[0][:int(n[0])]), int(n[0]), list(d[0])


def test_copy_continues():
    # t = 5 6 7 5 6 8 5 6 7 5 6.  Last 4-gram 6 7 5 6 occurs at 1 (next 8) -> 8;
    # then 7 5 6 8 at 2 (next 5) -> 5; then 5 6 8 5 at 3 (next 6) -> 6.
    assert draft1([5, 6, 7, 5, 6, 8, 5, 6, 7, 5, 6], 3)[:2] == ([8, 5, 6], 3)


def test_tie_goes_to_the_smaller_token_and_half_is_enough():
    # 1 2 3 4 occurs at 0 (next 9) and 5 (next 3): a tie, 3 wins; share 1/2 >= 1/2.
    # Then 2 3 4 3 at 6 (next 1) -> 1; 3 4 3 1 at 7 (next 2) -> 2.
    h = [1, 2, 3, 4, 9, 1, 2, 3, 4, 3, 1, 2, 3, 4]
    assert draft1(h, 3)[:2] == ([3, 1, 2], 3)
    # a 2/3 share: 1/2 fails at every n (each n-gram of the suffix has the same two
    # next tokens 9 and 3), so nothing is drafted.
    assert draft1(h, 3, share=[(2, 3)] * 4)[:2] == ([], 0)


def test_falls_back_to_a_shorter_ngram():
    # 1 2 3 4 is followed by 9, 3, 7 (share 1/3 < 1/2) and so are 2 3 4 and 3 4;
    # the 1-gram 4 is followed by 9, 3, 7, 7: 7 has 2 of 4 -> 7.  Then 2 3 4 7 at
    # 11 (next 8) -> 8; 3 4 7 8 at 12 (next 4) -> 4.
    h = [1, 2, 3, 4, 9, 1, 2, 3, 4, 3, 1, 2, 3, 4, 7, 8, 4, 7, 1, 2, 3, 4]
    assert draft1(h, 3)[:2] == ([7, 8, 4], 3)
    # restricted to n in 3..4 nothing passes.
    assert draft1(h, 3, n_min=3)[:2] == ([], 0)


def test_min_count():
    # with min_count 2 everywhere the 4- and 3-grams (one occurrence each) fail;
    # the 2-gram 5 6 occurs at 0, 3, 6 with next 7, 8, 7 -> 7 (2 of 3).  Then
    # 7 5 6 7 never occurred; 5 6 7 at 0 and 6 (next 5, 5) -> 5; 5 6 7 5 at 0
    # and 6 (next 6, 6) -> 6.
    assert draft1([5, 6, 7, 5, 6, 8, 5, 6, 7, 5, 6], 3, min_count=[2, 2, 2, 2])[:2] == ([7, 5, 6], 3)


def test_no_repeat_no_draft_and_sentinels():
    d, n, full = draft1(list(range(100, 140)), 5)
    assert (d, n, full) == ([], 0, [-1] * 5)


def test_short_histories():
    assert draft1([], 4)[1] == 0
    assert draft1([7], 4)[1] == 0                      # 7 has no earlier occurrence with a next token
    # 7 7: the 1-gram 7 occurred at 0 followed by 7; longer n-grams never occurred.
    assert draft1([7, 7], 4)[:2] == ([7, 7, 7, 7], 4)
    assert draft1([7, 7], 0)[:2] == ([], 0)


@pytest.mark.parametrize("d", [1, 2, 3, 7])
def test_periodic_closed_form(d):
    """Period-d history of distinct tokens: every n-gram has one next token, so
    the draft continues the period: draft[j] = a[(L + j) mod d]."""
    a = np.arange(d, dtype=np.int32) * 3 + 11
    L = d + 9
    t = a[np.arange(L) % d]
    K = 12
    dr, n, _ = draft1(list(t), K)
    assert n == K and dr == list(a[(L + np.arange(K)) % d])


def test_batch_matches_single_requests():
    # A CSR batch (offsets[0] > 0, an empty request) gives each request's own answer.
    hs = [[5, 6, 7, 5, 6, 8, 5, 6, 7, 5, 6], [], [7, 7], [1, 2, 3, 4, 9, 1, 2, 3, 4, 3, 1, 2, 3, 4]]
    lead = [42, 43, 44]
    tokens = np.array(lead + [x for h in hs for x in h], np.int32)
    offsets = len(lead) + gen.offsets_from_lengths([len(h) for h in hs])
    d, n = oracle.ctx_draft(tokens, offsets, 3)
    assert [list(d[r][:n[r]]) for r in range(4)] == [[8, 5, 6], [], [7, 7, 7], [3, 1, 2]]


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.ctx_draft(np.zeros(3, np.int32), np.array([0, 3]), 2, n_min=0)
    with pytest.raises(ValueError):
        oracle.ctx_draft(np.zeros(3, np.int32), np.array([0, 3]), 2, n_max=5)
    with pytest.raises(ValueError):
        oracle.ctx_draft(np.zeros(3, np.int32), np.array([0, 3]), 2, share=[(1, 0)] * 4)
