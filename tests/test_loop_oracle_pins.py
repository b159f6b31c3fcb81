"""Pins of the loop-step oracle (oracle/loop_oracle.c) against hand-worked cases.

Rules (HyperQwen lookup-drafting article, kwkr.cn/news/564408):
  "第2步"  head: a lookup match >= 8 replaces the draft model's proposals; >= 6 is
          adopted only if the model proposed the same first 2 tokens; tail: >= 4.
  "第3步"  long block entered when the match can fill the tail and the previous
          step's output was a nearly full block, two steps in a row; kept for 3
          steps after that drops.  Greedy verification accepts the agreeing
          prefix; a lookup position is a point mass on its token.
Every expected value below is worked out by hand from those rules (the working is
in the comments), not taken from any implementation.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

H, T = 3, 2
LOOKUP = [10, 11, 12, 13, 14, 15]            # K = 6 >= H + T


def fuse1(m, model, is_long, **kw):
    block, ln, pm = oracle.fuse([LOOKUP], [m], [model], [is_long], H, T, **kw)
    return list(block[0]), int(ln[0]), list(pm[0])


def test_fuse_long_match_replaces_head():
    # m = 8 >= replace_min: head = lookup; long and 8 >= 4: tail = lookup[3..5).
    assert fuse1(8, [10, 98, 99], 1) == ([10, 11, 12, 13, 14], 5, [1, 1, 1, 1, 1])


def test_fuse_shorter_match_needs_agreement():
    # m = 7 (>= 6, < 8): adopted when the model's first 2 tokens are 10, 11.
    assert fuse1(7, [10, 11, 99], 1) == ([10, 11, 12, 13, 14], 5, [1, 1, 1, 1, 1])
    # disagreement on the second token: the model's head stays; the tail (7 >= 4) is lookup's.
    assert fuse1(7, [10, 98, 99], 1) == ([10, 98, 99, 13, 14], 5, [0, 0, 0, 1, 1])
    # m = 6 with agreement, short block: head adopted, no tail.
    assert fuse1(6, [10, 11, 99], 0) == ([10, 11, 12, -1, -1], 3, [1, 1, 1, 0, 0])


def test_fuse_below_thresholds():
    # m = 5 < 6: even an agreeing model keeps its head; the tail needs only 4.
    assert fuse1(5, [10, 11, 99], 1) == ([10, 11, 99, 13, 14], 5, [0, 0, 0, 1, 1])
    # m = 4, exactly the tail threshold: the model's head, the lookup tail.
    assert fuse1(4, [7, 8, 9], 1) == ([7, 8, 9, 13, 14], 5, [0, 0, 0, 1, 1])
    # m = 3 < 4: nothing from lookup, even in a long step.
    assert fuse1(3, [7, 8, 9], 1) == ([7, 8, 9, -1, -1], 3, [0, 0, 0, 0, 0])
    # no match at all.
    assert fuse1(0, [7, 8, 9], 1) == ([7, 8, 9, -1, -1], 3, [0, 0, 0, 0, 0])


def test_fuse_agreement_width_zero():
    # agree_n = 0: any match >= agree_min is adopted.
    assert fuse1(6, [1, 2, 3], 0, agree_n=0) == ([10, 11, 12, -1, -1], 3, [1, 1, 1, 0, 0])


def test_fuse_no_long_flags_means_short():
    block, ln, pm = oracle.fuse([LOOKUP], [9], [[1, 2, 3]], None, H, T)
    assert list(ln) == [3] and list(block[0]) == [10, 11, 12, -1, -1]


def test_schedule_trace():
    """H = 7, T = 8: a full short block commits 8 tokens, a full long one 16;
    tail_min 4, slack 1 (nearly full = full - 1), enter after 2 steps, sticky 3.
      t1 (12, 8): short, full 8, cond (12>=4, 8>=7) yes, streak 1 -> 0
      t2 (12, 7): cond yes, streak 2 -> enter, hold 3 -> 1
      t3 (12,16): long, full 16, 16>=15 yes, hold 3 -> 1
      t4 ( 2,16): m < 4, no: hold 3->2 -> 1
      t5 (12, 3): 3 < 15, no: hold 2->1 -> 1
      t6 (12,14): 14 < 15, no: hold 1->0 -> 1
      t7 ( 0,16): no, hold 0: exit -> 0
      t8 (12, 8): short again, full 8, yes, streak 1 -> 0
      t9 (12, 6): 6 < 7, no, streak 0 -> 0
     t10 (12, 8): yes, streak 1 -> 0
     t11 (12, 8): yes, streak 2 -> enter -> 1"""
    steps = [(12, 8), (12, 7), (12, 16), (2, 16), (12, 3), (12, 14), (0, 16), (12, 8), (12, 6),
             (12, 8), (12, 8)]
    want = [0, 1, 1, 1, 1, 1, 0, 0, 0, 0, 1]
    state = np.zeros((1, 3), np.int32)
    got = [int(oracle.schedule([m], [c], state, 7, 8)[0]) for m, c in steps]
    assert got == want


def test_schedule_threshold_boundaries():
    """m exactly tail_min (4) counts; committed exactly full - slack (7 of 8) counts;
    one less of either does not.
      (4, 7) yes streak 1; (4, 7) yes streak 2 -> enter;  a second request:
      (3, 8) no; (4, 6) no; (4, 7) yes streak 1; (4, 7) yes streak 2 -> enter."""
    state = np.zeros((1, 3), np.int32)
    got = [int(oracle.schedule([m], [c], state, 7, 8)[0]) for m, c in [(4, 7), (4, 7)]]
    assert got == [0, 1]
    state = np.zeros((1, 3), np.int32)
    got = [int(oracle.schedule([m], [c], state, 7, 8)[0]) for m, c in [(3, 8), (4, 6), (4, 7), (4, 7)]]
    assert got == [0, 0, 0, 1]


def test_schedule_requests_are_independent():
    state = np.zeros((2, 3), np.int32)
    outs = [oracle.schedule([12, 0], [8, 8], state, 7, 8) for _ in range(2)]
    assert [list(o) for o in outs] == [[0, 0], [1, 0]]


def test_verify_greedy():
    # block 5 6 7 8, target 5 6 9 ...: agree on 2 tokens, commit 5 6 then the target's 9.
    acc, commit, nc = oracle.verify([[5, 6, 7, 8]], [4], [[5, 6, 9, 8, 1]])
    assert (int(acc[0]), list(commit[0]), int(nc[0])) == (2, [5, 6, 9, -1, -1], 3)
    # all of len = 2 accepted: commit both, then the target's token at position 2.
    acc, commit, nc = oracle.verify([[5, 6, -1, -1]], [2], [[5, 6, 7, 0, 0]])
    assert (int(acc[0]), list(commit[0]), int(nc[0])) == (2, [5, 6, 7, -1, -1], 3)
    # nothing proposed: commit the target's first token.
    acc, commit, nc = oracle.verify([[1, 2, 3, 4]], [0], [[9, 9, 9, 9, 9]])
    assert (int(acc[0]), list(commit[0]), int(nc[0])) == (0, [9, -1, -1, -1, -1], 1)


def test_verify_sampled_and_point_mass():
    block, ln, target = [[5, 6, 7]], [3], [[50, 60, 70, 80]]
    p = [[0.5, 0.9, 0.2]]
    q = [[1.0, 0.5, 0.1]]
    u = [[0.4, 0.95, 0.3]]
    # 0.4*1 < 0.5, 0.95*0.5 = 0.475 < 0.9, 0.3*0.1 = 0.03 < 0.2: all accepted, bonus 80.
    acc, commit, nc = oracle.verify(block, ln, target, probs=p, qprobs=q, u=u)
    assert (int(acc[0]), list(commit[0])) == (3, [5, 6, 7, 80])
    # position 1 filled by lookup: a point mass, q = 1; 0.95*1 < 0.9 fails: commit 5, 60.
    acc, commit, nc = oracle.verify(block, ln, target, probs=p, qprobs=q, u=u, point_mass=[[0, 1, 0]])
    assert (int(acc[0]), list(commit[0]), int(nc[0])) == (1, [5, 60, -1, -1], 2)


def test_append_is_concatenation():
    rng = np.random.default_rng(0)
    lengths = [0, 3, 5, 0, 2]
    lead = 4
    tokens = rng.integers(0, 100, size=lead + sum(lengths)).astype(np.int32)
    offsets = lead + np.concatenate([[0], np.cumsum(lengths)])
    commit = rng.integers(100, 200, size=(5, 4)).astype(np.int32)
    ncommit = np.array([1, 4, 0, 2, 3], np.int32)
    out_t, out_o = oracle.append(tokens, offsets, commit, ncommit)
    hist = []
    for r in range(5):
        hist.append(list(tokens[offsets[r]:offsets[r + 1]]) + list(commit[r][:ncommit[r]]))
    assert list(out_o) == list(np.concatenate([[0], np.cumsum([len(h) for h in hist])]))
    assert list(out_t) == [x for h in hist for x in h]


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.fuse([LOOKUP], [8], [[1, 2, 3]], [1], 4, 3)      # K < H + T
    with pytest.raises(ValueError):
        oracle.verify([[1, 2]], [3], [[1, 2, 3]])               # len > P
