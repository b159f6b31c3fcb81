"""GPU parity of context-cache drafting (include/lookup_ctxcache.h) with the oracle.

Exact comparison of every draft token and length, after a build and after every
append of a decode loop, for several thresholds and n ranges, on the workloads
and on small-alphabet streams where ties and thresholds decide often -- also
with token values anywhere in int32 (negative, at or beyond 2^20, INT32_MIN and
INT32_MAX), which the cache keys through its dictionary of codes, and with
ties between negative and positive tokens.  A cache whose dictionary runs out of
codes must fail its requests, never draft from incomplete counts.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle

torch = pytest.importorskip("torch")
pkg = pytest.importorskip("prompt_lookup_speculative_gb300")

pytestmark = pytest.mark.gpu

SHARE_HALF = ((1, 2),) * 4


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def setup(tokens, offsets, spare, seed, n_min=1, n_max=4, **kw):
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, spare, seed=seed)
    t, b, n = dev(st), dev(base), dev(length)
    cc = pkg.ContextCache(st.shape[0], n_min, n_max, **kw)
    cc.build(t, b, n)
    return cc, st, base, length, cap, t, b, n


def check(cc, t, b, n, tokens, offsets, K, n_min=1, n_max=4, min_count=(1, 1, 1, 1), share=SHARE_HALF):
    d, ln = cc.draft(t, b, n, K)
    wd, wl = oracle.ctx_draft(tokens, offsets, K, n_min=n_min, n_max=n_max, min_count=min_count, share=share,
                              threads=16)
    np.testing.assert_array_equal(host(ln), wl)
    np.testing.assert_array_equal(host(d), wd)
    return wl


@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_ctx_draft_matches_oracle(name):
    w = gen.make_workload(name)
    cc, st, base, length, cap, t, b, n = setup(w.tokens, w.offsets, 16, w.seed)
    lens = check(cc, t, b, n, w.tokens, w.offsets, 8)
    if name in ("tiny", "recitation25k", "periodic"):
        assert lens.sum() > 0


def small_alphabet_batch(seed, B=200, vocab=6, Lmax=400):
    rng = gen.rng_for(seed, 61)
    lengths = rng.integers(0, Lmax, size=B)
    tokens = rng.integers(0, vocab, size=int(lengths.sum())).astype(np.int32)
    return tokens, gen.offsets_from_lengths(lengths)


@pytest.mark.parametrize("params", [
    dict(),
    dict(min_count=(2, 2, 2, 2)),
    dict(min_count=(5, 3, 2, 1), share=((2, 3), (3, 5), (1, 2), (1, 1))),
    dict(share=((0, 1),) * 4),
    dict(n_min=2, n_max=3),
    dict(n_min=4, n_max=4),
    dict(n_min=1, n_max=1),
])
@pytest.mark.parametrize("vocab", [2, 6, 40])
def test_ctx_thresholds_and_ranges(params, vocab):
    tokens, offsets = small_alphabet_batch(vocab, vocab=vocab)
    n_min, n_max = params.get("n_min", 1), params.get("n_max", 4)
    mc = params.get("min_count", (1, 1, 1, 1))
    share = params.get("share", SHARE_HALF)
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 0, 2, n_min, n_max, min_count=mc, share=share)
    check(cc, t, b, n, tokens, offsets, 12, n_min, n_max, mc, share)


@pytest.mark.parametrize("K", [0, 1, 64])
def test_ctx_draft_lengths(K):
    tokens, offsets = small_alphabet_batch(7, vocab=3)
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 0, 3)
    check(cc, t, b, n, tokens, offsets, K)


@pytest.mark.parametrize("name,vocab", [("tiny", None), ("chats", None), ("small", 4)])
def test_ctx_decode_loop(name, vocab):
    """Draft, commit a synthetic continuation (an accepted prefix of the draft,
    then one more token), append in place, compare with the oracle each step."""
    if name == "small":
        tokens, offsets = small_alphabet_batch(11, B=300, vocab=vocab)
    else:
        w = gen.make_workload(name)
        tokens, offsets = w.tokens, w.offsets
    B = offsets.shape[0] - 1
    W, K = 9, 8
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 6 * W, 4)
    capd = dev(cap)
    rng = gen.rng_for(B, 62)
    cur_t, cur_o = tokens, offsets
    for step in range(5):
        d, ln = cc.draft(t, b, n, K)
        wd, wl = oracle.ctx_draft(cur_t, cur_o, K, threads=16)
        np.testing.assert_array_equal(host(ln), wl)
        np.testing.assert_array_equal(host(d), wd)
        acc = np.minimum(rng.integers(0, K + 1, size=B), wl)
        commit = rng.integers(0, vocab or 50, size=(B, W)).astype(np.int32)
        for r in range(B):
            commit[r, :acc[r]] = wd[r, :acc[r]]
        ncommit = (acc + 1).astype(np.int32)
        assert (host(cc.append(t, b, n, capd, dev(commit), dev(ncommit))) == 0).all()
        cur_t, cur_o = oracle.append(cur_t, cur_o, commit, ncommit)
        got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
        np.testing.assert_array_equal(got_o, cur_o)
        np.testing.assert_array_equal(got_t, cur_t)


def test_ctx_status_mismatch_and_overflow():
    tokens, offsets = small_alphabet_batch(13, B=20, vocab=5)
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 3, 5)
    commit = np.arange(20 * 5, dtype=np.int32).reshape(20, 5) % 5
    ncommit = np.array([4, 3] * 10, np.int32)                      # 4 does not fit in 3 spare slots
    status = host(cc.append(t, b, n, dev(cap), dev(commit), dev(ncommit)))
    assert list(status) == [1, 0] * 10
    # a cache queried with other lengths fails its requests
    other = pkg.ContextCache(10, 2, 4, slots=cc.slots)
    other.memory = cc.memory
    d, ln = other.draft(t, b, n, 4)
    assert (host(ln) == pkg.LEN_FAILED).all()
    # a table far too small overflows: every request reports the failure
    small = pkg.ContextCache(st.shape[0], 1, 4, slots=64)
    small.build(t, b, n)
    d, ln = small.draft(t, b, n, 4)
    assert (host(ln) == pkg.LEN_FAILED).all()


@pytest.mark.parametrize("B", [300, 12000])
def test_ctx_append_both_launch_shapes(B):
    """The append runs one CTA per request when the batch fits in one wave of
    them, else dense tasks then a length pass: same tokens, lengths, statuses and
    next drafts either way."""
    rng = np.random.default_rng(B + 7)
    lengths = rng.integers(0, 60, size=B)
    tokens = rng.integers(0, 6, size=int(lengths.sum())).astype(np.int32)
    offsets = gen.offsets_from_lengths(lengths)
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 4, seed=B)
    t, b, n = dev(st), dev(base), dev(length)
    cc = pkg.ContextCache(st.shape[0], 1, 4)
    cc.build(t, b, n)
    W = 6
    commit = rng.integers(0, 6, size=(B, W)).astype(np.int32)
    ncommit = rng.integers(0, W + 1, size=B).astype(np.int32)      # 5 and 6 do not fit in 4 spare slots
    status = host(cc.append(t, b, n, dev(cap), dev(commit), dev(ncommit)))
    fits = ncommit <= 4
    np.testing.assert_array_equal(status, np.where(fits, 0, 1))
    np.testing.assert_array_equal(host(n), length + np.where(fits, ncommit, 0))
    want_t, want_o = oracle.append(tokens, offsets, commit, np.where(fits, ncommit, 0).astype(np.int32))
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_o, want_o)
    np.testing.assert_array_equal(got_t, want_t)
    d, ln = cc.draft(t, b, n, 5)
    wd, wl = oracle.ctx_draft(want_t, want_o, 5, threads=16)
    np.testing.assert_array_equal(host(ln), wl)
    np.testing.assert_array_equal(host(d), wd)


# Token values that are not their own code in the cache's keys, and a few that are.
WIDE_VALUES = np.array([-(2**31), 2**31 - 1, -1, -2, -7, 2**20, 2**20 + 1, 2**21, 2**30 + 3, -(2**20),
                        0, 1, 5, 2**20 - 1], dtype=np.int64)


def wide_alphabet_batch(seed, B=200, vocab=6, Lmax=400):
    """Small-alphabet histories whose letters are drawn from WIDE_VALUES."""
    rng = gen.rng_for(seed, 63)
    letters = rng.choice(WIDE_VALUES, size=vocab, replace=False)
    lengths = rng.integers(0, Lmax, size=B)
    tokens = letters[rng.integers(0, vocab, size=int(lengths.sum()))].astype(np.int32)
    return tokens, gen.offsets_from_lengths(lengths), letters


@pytest.mark.parametrize("params", [dict(), dict(n_min=2, n_max=3), dict(n_min=1, n_max=1),
                                    dict(min_count=(2, 2, 2, 2), share=((2, 3),) * 4)])
@pytest.mark.parametrize("vocab", [2, 3, 6, 14])
def test_ctx_any_int32_tokens(params, vocab):
    tokens, offsets, letters = wide_alphabet_batch(vocab * 10 + len(params), vocab=vocab)
    assert (letters < 0).any() or (letters >= 2**20).any()
    n_min, n_max = params.get("n_min", 1), params.get("n_max", 4)
    mc = params.get("min_count", (1, 1, 1, 1))
    share = params.get("share", SHARE_HALF)
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 0, 6, n_min, n_max, min_count=mc, share=share)
    lens = check(cc, t, b, n, tokens, offsets, 12, n_min, n_max, mc, share)
    assert lens.sum() > 0


def test_ctx_ties_follow_signed_order():
    """Equal counts go to the smallest signed token: a history where INT32_MIN, -1,
    0 and INT32_MAX each follow the same 1-gram once (the oracle drafts
    INT32_MIN), and one without INT32_MIN (it drafts -1)."""
    a = 77
    body = [a, 2**31 - 1, a, 0, a, -1, a, -(2**31), a]
    body2 = [a, 2**31 - 1, a, 0, a, -1, a, 5, a]
    tokens = np.array(body + body2, dtype=np.int32)
    offsets = np.array([0, len(body), len(body) + len(body2)], dtype=np.int64)
    any_share = ((0, 1),) * 4                              # every candidate passes the share test
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 0, 7, 1, 1, share=any_share)
    d, ln = cc.draft(t, b, n, 1)
    assert list(host(d)[:, 0]) == [-(2**31), -1]
    check(cc, t, b, n, tokens, offsets, 1, 1, 1, share=any_share)


def test_ctx_decode_loop_any_int32_tokens():
    """The decode loop of test_ctx_decode_loop with wide token values, committed
    tokens included: the appends give new values codes as they arrive."""
    tokens, offsets, letters = wide_alphabet_batch(71, B=150, vocab=5)
    B = offsets.shape[0] - 1
    W, K = 9, 8
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 6 * W, 8)
    capd = dev(cap)
    rng = gen.rng_for(B, 64)
    pool = np.concatenate([letters, [-5, 2**20 + 9, 2**31 - 2]]).astype(np.int64)
    cur_t, cur_o = tokens, offsets
    for step in range(5):
        d, ln = cc.draft(t, b, n, K)
        wd, wl = oracle.ctx_draft(cur_t, cur_o, K, threads=16)
        np.testing.assert_array_equal(host(ln), wl)
        np.testing.assert_array_equal(host(d), wd)
        acc = np.minimum(rng.integers(0, K + 1, size=B), wl)
        commit = pool[rng.integers(0, pool.size, size=(B, W))].astype(np.int32)
        for r in range(B):
            commit[r, :acc[r]] = wd[r, :acc[r]]
        ncommit = (acc + 1).astype(np.int32)
        assert (host(cc.append(t, b, n, capd, dev(commit), dev(ncommit))) == 0).all()
        cur_t, cur_o = oracle.append(cur_t, cur_o, commit, ncommit)


def test_ctx_out_of_codes_fails_every_request():
    """More distinct values outside [0, 2^20) than the dictionary has codes: the
    drafts report LOOKUP_DRAFT_LEN_FAILED rather than drafting from incomplete
    counts."""
    n_vals = 2**20 + 4096
    vals = -(np.arange(n_vals, dtype=np.int64) + 1)          # all distinct, all negative
    tokens = np.concatenate([vals, vals[:64]]).astype(np.int32)
    offsets = np.array([0, n_vals // 2, tokens.size], dtype=np.int64)
    cc, st, base, length, cap, t, b, n = setup(tokens, offsets, 0, 9, 1, 1)
    d, ln = cc.draft(t, b, n, 4)
    assert (host(ln) == pkg.LEN_FAILED).all()
