"""The seeded input generators' options (gen/): a resized recitation batch.

The size sweep of the benchmark runs the recitation recipe at other history
lengths.  With its default length the override must give the default batch
draw for draw, and in a resized batch the planted copies must sit where the
construction puts them (checked with the oracle, as the planted-copy pins do).
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle


def test_recitation_length_override_keeps_the_recipe():
    a = gen.make_workload("recitation25k")
    b = gen.make_workload("recitation25k", length=25000)
    np.testing.assert_array_equal(a.tokens, b.tokens)
    np.testing.assert_array_equal(a.offsets, b.offsets)
    assert a.planted == b.planted and (a.min_m, a.max_m, a.K) == (b.min_m, b.max_m, b.K)
    assert b.name == "recitation_L25000"


@pytest.mark.parametrize("name,length", [("recitation25k", 4000), ("recitation25k", 0), ("chats", 8192)])
def test_recitation_length_is_checked(name, length):
    with pytest.raises(ValueError):
        gen.make_workload(name, length=length)


@pytest.mark.parametrize("length", [4096, 8192])
def test_resized_recitation_planted_copies(length):
    """A planted request ends in a copy of t[s0 : s0+c]; for c >= 12 its 12-suffix is
    t[s0+c-12 : s0+c], so m = 12 and p = s0 + c - 12 (a Zipf text repeating 12
    tokens elsewhere by chance is far less likely than the planted copy)."""
    w = gen.make_workload("recitation25k", length=length)
    assert w.B == 64 and w.total_tokens == 64 * length and w.planted
    draft, ln, pos, m = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=4)
    checked = 0
    for r, (s0, c) in w.planted.items():
        if c < 12:
            continue
        t = w.tokens[w.offsets[r]:w.offsets[r + 1]]
        assert (m[r], pos[r], ln[r]) == (12, s0 + c - 12, 15), r
        np.testing.assert_array_equal(draft[r], t[s0 + c:s0 + c + 15])
        checked += 1
    assert checked >= 5
