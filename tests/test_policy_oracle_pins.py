"""Pins of the draft-source controller oracle (oracle/policy_oracle.c).

Rule (Strata engine article, gtnt.cn/news/124732, section 五): every step, for the
draft model's draft and the lookup draft, estimate E[committed tokens] / verify
time; the acceptance rate is an EMA kept per match-length bucket (four) for the
lookup draft; use the lookup draft only when its benefit exceeds the model's by
more than the margin; fall back to plain decoding when speculation does not pay.
The readings the oracle takes (E = 1 + a + ... + a^n, the EMA, the bucket edges)
are stated in its header.

Every expected value below is worked out by hand in the comments, with numbers
that are exact in binary floating point, so the comparisons are exact.
"""
from __future__ import annotations

import numpy as np

import oracle

# t_lookup = 1, t_model = 1.25, t_plain = 1, alpha = 1/4, margin = 1/4 unless stated
BASE = dict(n_lookup=4, n_model=3, t_lookup=1.0, t_model=1.25, t_plain=1.0, alpha=0.25, margin=0.25)


def state(B=1, a=0.5):
    return np.full((B, 5), a, np.float32), np.zeros((B, 3), np.int32)


def step(m, accepted, acc, prev, **kw):
    args = dict(BASE)
    args.update(kw)
    return list(oracle.policy(np.atleast_1d(m), np.atleast_1d(accepted), acc, prev, **args))


def test_lookup_wins_by_more_than_the_margin():
    # model: E(0.5, 3) = 1 + .5 + .25 + .125 = 1.875, / 1.25 = 1.5; x (1 + 1/4) = 1.875.
    # lookup (m = 12, bucket 3): E(0.5, 4) = 1.9375, / 1 = 1.9375 > 1.875 -> lookup;
    # plain 1 / 1 = 1 < 1.9375.
    acc, prev = state()
    assert step(12, 0, acc, prev) == [2]
    assert list(prev[0]) == [2, 3, 4]                    # choice, bucket, tokens drafted


def test_a_tie_with_the_margin_keeps_the_model():
    # n_lookup = 3: E = 1.875 = exactly 1.25 x 1.5, not more -> the model (1), and
    # 1.5 > plain's 1.
    acc, prev = state()
    assert step(12, 0, acc, prev, n_lookup=3) == [1]
    assert list(prev[0]) == [1, 0, 3]


def test_no_match_means_no_lookup():
    # m = 0: the lookup draft does not exist; model 1.5 > plain 1 -> model.
    acc, prev = state()
    assert step(0, 0, acc, prev) == [1]


def test_plain_decoding_when_speculation_does_not_pay():
    # t_plain = 0.5: plain commits 1 / 0.5 = 2 per unit; lookup 1.9375 and model 1.5
    # are both below -> plain (0), nothing drafted.
    acc, prev = state()
    assert step(12, 0, acc, prev, t_plain=0.5) == [0]
    assert list(prev[0]) == [0, 0, 0]
    # t_plain = 0.5625 (1 / 0.5625 = 1.777...): the lookup's 1.9375 beats it.
    acc, prev = state()
    assert step(12, 0, acc, prev, t_plain=0.5625) == [2]
    # lookup's benefit exactly plain's: 1 / t_plain = 1.9375 needs t_plain = 16/31
    # (not exact); use E = 2 instead: a = 1 gives E(1, 1) = 2 with n_lookup = 1, and
    # t_plain = 0.5 -> 2 == 2, not more -> plain.
    acc, prev = state(a=1.0)
    assert step(12, 0, acc, prev, n_lookup=1, n_model=0, t_plain=0.5) == [0]


def test_buckets_of_the_match_length():
    # edges (6, 8, 12): m 4, 5 -> 0; 6, 7 -> 1; 8..11 -> 2; 12 and above -> 3.  Give
    # the four buckets acceptances 0, 0, 0, 1 with n_lookup = 1: E = 1 in buckets 0-2
    # (lookup 1 < 1.875) and E = 2 in bucket 3 (2 > 1.875).
    for m, want in ((4, 1), (5, 1), (6, 1), (7, 1), (8, 1), (11, 1), (12, 2), (13, 2)):
        acc = np.array([[0.0, 0.0, 0.0, 1.0, 0.5]], np.float32)
        prev = np.zeros((1, 3), np.int32)
        assert step(m, 0, acc, prev, n_lookup=1) == [want], m
    # the recorded bucket after a lookup choice
    for m, b in ((4, 0), (6, 1), (7, 1), (8, 2), (11, 2), (12, 3)):
        acc = np.array([[1.0, 1.0, 1.0, 1.0, 0.0]], np.float32)
        prev = np.zeros((1, 3), np.int32)
        assert step(m, 0, acc, prev, n_lookup=1) == [2], m
        assert prev[0, 1] == b, m


def test_ema_update_goes_to_the_source_and_bucket_that_drafted():
    # step 1: lookup chosen in bucket 3 with 4 tokens (as above).
    acc, prev = state()
    assert step(12, 0, acc, prev) == [2]
    # step 2: 4 of 4 accepted -> rate 1; acc[3] = 0.75 x 0.5 + 0.25 x 1 = 0.625; the
    # other slots keep 0.5.
    step(5, 4, acc, prev)
    assert list(acc[0]) == [0.5, 0.5, 0.5, 0.625, 0.5]
    # step 2's own choice: m = 5 is bucket 0, E(0.5, 4) = 1.9375 > 1.875 -> lookup, bucket 0.
    assert list(prev[0]) == [2, 0, 4]
    # step 3: 1 of 4 accepted -> rate 0.25; acc[0] = 0.375 + 0.0625 = 0.4375.
    step(0, 1, acc, prev)
    assert list(acc[0]) == [0.4375, 0.5, 0.5, 0.625, 0.5]
    # step 3's choice: no match -> model, 3 tokens.
    assert list(prev[0]) == [1, 0, 3]
    # step 4: 0 of 3 accepted -> the model's acc[4] = 0.375 + 0 = 0.375.
    step(0, 0, acc, prev)
    assert list(acc[0]) == [0.4375, 0.5, 0.5, 0.625, 0.375]


def test_no_update_after_plain_decoding_or_a_first_step():
    acc, prev = state()
    step(12, 3, acc, prev, t_plain=0.5)                  # first step: nothing to update; plain chosen
    assert list(acc[0]) == [0.5] * 5
    step(12, 3, acc, prev, t_plain=0.5)                  # after plain: nothing drafted, nothing to update
    assert list(acc[0]) == [0.5] * 5


def test_accepted_is_clamped_to_the_drafted_tokens():
    acc, prev = state()
    step(12, 0, acc, prev)                               # lookup, bucket 3, 4 tokens
    step(12, 9, acc, prev)                               # 9 > 4 counts as 4: rate 1 -> 0.625
    assert acc[0, 3] == np.float32(0.625)
    step(12, -2, acc, prev)                              # -2 counts as 0: 0.75 x 0.625 = 0.46875
    assert acc[0, 3] == np.float32(0.46875)


def test_requests_are_independent():
    acc, prev = state(B=3)
    acc[1] = [1.0, 1.0, 1.0, 1.0, 0.0]
    got = oracle.policy(np.array([12, 12, 0]), np.zeros(3, np.int32), acc, prev, **BASE)
    # request 0 as in the first test; request 1: model E(0, 3) = 1 -> 0.8, lookup E(1, 4)
    # = 5 -> lookup; request 2: no match, model 1.5 -> model.
    assert list(got) == [2, 2, 1]


def test_rejects_bad_parameters():
    acc, prev = state()
    for bad in (dict(t_model=0.0), dict(t_plain=-1.0), dict(alpha=1.5), dict(margin=-0.1), dict(n_model=-1),
                dict(edges=(8, 6, 12))):
        args = dict(BASE)
        args.update(bad)
        try:
            oracle.policy([12], [0], acc, prev, **args)
        except ValueError:
            continue
        raise AssertionError(f"accepted {bad}")
