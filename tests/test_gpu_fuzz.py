"""Randomised parity sweeps of the drafting step against the oracle.

Every case is drawn from a seeded generator, so a failure names a reproducible
case.  A case mixes what the fixed tests take one at a time:
- batch sizes from 1 to 6,000 requests (both fills, offsets in shared and in
  global memory);
- history lengths from empty through short (under min_m) to 60,000 tokens;
- alphabets from 2 letters (dense matches, periodic text) to a Zipf vocabulary,
  with some tokens replaced by INT32_MIN, INT32_MAX and negative values;
- m ranges anywhere in [1, 32], K in [0, 64], every 4-byte phase of the tokens
  pointer, and tokens before offsets[0] that belong to no request.
Each case is compared element by element with the oracle: the draft, its
length, the position and m.  The two-launch loop path (draft, then scheduling
and fusion) is swept the same way against the oracle's draft, schedule and fuse,
and the incremental index and the context cache over random 3-step decode loops
(draft, commit, append in place), the index also in its two-launch form (draft
with scheduling and fusion, then verification with the append) and in plain
prompt-lookup decoding (verification, append and the next draft in one launch).
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytestmark = [pytest.mark.gpu, pytest.mark.skip(reason="needs a CUDA GPU")]

import prompt_lookup_speculative_gb300 as pkg  # noqa: E402

DEV = "cuda:0"
EXTREMES = np.array([np.iinfo(np.int32).min, np.iinfo(np.int32).max, -1, -7, 1 << 20], np.int32)


def random_batch(rng: np.random.Generator):
    """A seeded random batch: (tokens, offsets, min_m, max_m, K, pad)."""
    B = int(np.exp(rng.uniform(0, np.log(6000))))
    kind = rng.integers(0, 4)
    if kind == 0:                                        # many short requests, some empty
        lengths = rng.integers(0, 40, size=B)
    elif kind == 1:                                      # log-uniform up to 60k
        lengths = np.exp(rng.uniform(0, np.log(60000), size=B)).astype(np.int64)
    elif kind == 2:                                      # a mixture with empties and near-min_m ones
        lengths = rng.choice([0, 1, 2, 3, 4, 5, 13, 200, 3000], size=B)
    else:                                                # equal lengths
        lengths = np.full(B, int(rng.integers(1, 5000)))
    budget = 3_000_000                                   # keep the oracle's work bounded
    if lengths.sum() > budget:
        lengths = (lengths * (budget / lengths.sum())).astype(np.int64)
    n = int(lengths.sum())
    alpha = int(rng.choice([2, 3, 5, 50, 32000]))
    if alpha == 32000:
        tokens = gen.zipf_tokens(rng, n, 32000, 1.1, rng.permutation(32000).astype(np.int32))
    else:
        tokens = rng.integers(0, alpha, size=n).astype(np.int32)
    if n and rng.random() < 0.3:                         # extreme values sprinkled in
        at = rng.integers(0, n, size=max(1, n // 50))
        tokens[at] = EXTREMES[rng.integers(0, EXTREMES.size, size=at.size)]
    lead = int(rng.integers(0, 10))
    tokens = np.concatenate([rng.integers(0, 3, lead).astype(np.int32), tokens])
    offsets = gen.offsets_from_lengths(lengths) + lead
    min_m = int(rng.integers(1, 9))
    max_m = int(rng.integers(min_m, 33))
    K = int(rng.integers(0, 65))
    pad = int(rng.integers(0, 4))
    return tokens.astype(np.int32), offsets.astype(np.int64), min_m, max_m, K, pad


def device_batch(tokens, offsets, pad):
    buf = torch.zeros(tokens.size + pad + 4, dtype=torch.int32, device=DEV)
    buf[pad:pad + tokens.size] = torch.from_numpy(tokens).to(DEV)
    return buf[pad:pad + tokens.size], torch.from_numpy(offsets).to(DEV)


@pytest.mark.parametrize("block", range(16))
def test_draft_matches_oracle_on_random_batches(block):
    """Sixteen blocks of 25 random cases each."""
    rng = np.random.default_rng(20260 + block)
    for case in range(25):
        tokens, offsets, min_m, max_m, K, pad = random_batch(rng)
        t, o = device_batch(tokens, offsets, pad)
        d, ln, p, m = pkg.lookup_draft_ex(t, o, min_m, max_m, K)
        torch.cuda.synchronize()
        want = oracle.lookup_draft(tokens, offsets, min_m, max_m, K, threads=16)
        label = (f"block {block} case {case}: B={offsets.size - 1} tokens={tokens.size} "
                 f"m=[{min_m},{max_m}] K={K} pad={pad}")
        for name, g, w in zip(("draft", "len", "pos", "mlen"), (d, ln, p, m), want):
            np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=f"{label}: {name}")


@pytest.mark.parametrize("block", range(6))
def test_draft_plan_matches_oracle_on_random_batches(block):
    """lookup_draft_plan on random batches, block shapes and thresholds, against
    the oracle's draft (K = H + T), schedule and fuse."""
    rng = np.random.default_rng(30260 + block)
    for case in range(25):
        tokens, offsets, min_m, max_m, _, pad = random_batch(rng)
        B = offsets.size - 1
        H = int(rng.integers(1, 33))
        T = int(rng.integers(0, 65 - H))
        agree_n = int(rng.integers(0, H + 1))
        kw = dict(replace_min=int(rng.integers(1, 13)), agree_min=int(rng.integers(1, 13)), agree_n=agree_n,
                  tail_min=int(rng.integers(1, 13)), slack=int(rng.integers(0, 4)),
                  enter_steps=int(rng.integers(1, 4)), sticky=int(rng.integers(0, 5)))
        d_o, l_o, p_o, m_o = oracle.lookup_draft(tokens, offsets, min_m, max_m, H + T, threads=16)
        md = rng.integers(-2, 4, size=(B, H)).astype(np.int32)
        take = rng.random(B) < 0.5
        md[take] = d_o[take, :H]
        committed = rng.integers(1, H + T + 2, size=B).astype(np.int32)
        state = np.stack([rng.integers(0, 2, B), rng.integers(0, 3, B), rng.integers(0, 4, B)], 1).astype(np.int32)
        st_o = state.copy()
        lg_o = oracle.schedule(m_o, committed, st_o, H, T, tail_min=kw["tail_min"], slack=kw["slack"],
                               enter_steps=kw["enter_steps"], sticky=kw["sticky"])
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T, replace_min=kw["replace_min"],
                                         agree_min=kw["agree_min"], agree_n=agree_n, tail_min=kw["tail_min"])
        t, o = device_batch(tokens, offsets, pad)
        st_g = torch.from_numpy(state.copy()).to(DEV)
        got = pkg.lookup_draft_plan(t, o, torch.from_numpy(md).to(DEV), torch.from_numpy(committed).to(DEV), st_g,
                                    min_m, max_m, H, T, **kw)
        torch.cuda.synchronize()
        label = f"block {block} case {case}: B={B} m=[{min_m},{max_m}] H={H} T={T} {kw}"
        for name, g, w in zip(("long", "block", "len", "point mass", "mlen", "draft len", "state"),
                              (*got, st_g), (lg_o, blk_o, len_o, pm_o, m_o, l_o, st_o)):
            np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=f"{label}: {name}")


def small_random_batch(rng: np.random.Generator):
    """A random batch kept small enough for the slab structures' memory: up to
    400 requests of up to 20,000 tokens, about 400k tokens at most."""
    B = int(np.exp(rng.uniform(0, np.log(400))))
    lengths = np.where(rng.random(B) < 0.2, rng.integers(0, 6, size=B),
                       np.exp(rng.uniform(0, np.log(20000), size=B)).astype(np.int64))
    if lengths.sum() > 400_000:
        lengths = (lengths * (400_000 / lengths.sum())).astype(np.int64)
    n = int(lengths.sum())
    alpha = int(rng.choice([2, 3, 7, 50, 32000]))
    tokens = rng.integers(0, alpha, size=n).astype(np.int32)
    if n and rng.random() < 0.3:
        at = rng.integers(0, n, size=max(1, n // 50))
        tokens[at] = EXTREMES[rng.integers(0, EXTREMES.size, size=at.size)]
    return tokens, gen.offsets_from_lengths(lengths).astype(np.int64)


def _commit(rng, draft, length, B, W, K):
    """A synthetic continuation: an accepted prefix of the draft, then one more token."""
    acc = np.minimum(rng.integers(0, W, size=B), np.where(length > 0, K, 0))
    commit = rng.integers(-3, 50, size=(B, W)).astype(np.int32)
    for r in range(B):
        commit[r, :acc[r]] = draft[r, :acc[r]]
    return commit, (acc + 1).astype(np.int32)


@pytest.mark.parametrize("case", range(12))
def test_index_matches_oracle_on_random_decode_loops(case):
    rng = np.random.default_rng(40260 + case)
    tokens, offsets = small_random_batch(rng)
    B = offsets.size - 1
    min_m = int(rng.integers(1, 7))
    max_m = int(rng.integers(min_m, 33))
    K = int(rng.integers(0, 65))
    W = 16
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 4 * W, seed=case)
    t, b, n = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (st, base, length))
    capd = torch.from_numpy(cap).to(DEV)
    idx = pkg.NgramIndex(st.shape[0], min_m, max_m)
    idx.build(t, b, n)
    cur_t, cur_o = tokens, offsets
    for step in range(3):
        d, ln, p, m = idx.draft(t, b, n, K)[:4]
        want = oracle.lookup_draft(cur_t, cur_o, min_m, max_m, K, threads=16)
        label = f"case {case} step {step}: B={B} m=[{min_m},{max_m}] K={K}"
        for name, g, w in zip(("draft", "len", "pos", "mlen"), (d, ln, p, m), want):
            np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=f"{label}: {name}")
        commit, ncommit = _commit(rng, want[0], want[1], B, W, K)
        status = idx.append(t, b, n, capd, torch.from_numpy(commit).to(DEV), torch.from_numpy(ncommit).to(DEV))
        assert (status.cpu().numpy() == 0).all(), label
        cur_t, cur_o = oracle.append(cur_t, cur_o, commit, ncommit)
        got_t, got_o = gen.csr_of_slabs(t.cpu().numpy(), base, n.cpu().numpy())
        np.testing.assert_array_equal(got_o, cur_o, err_msg=label)
        np.testing.assert_array_equal(got_t, cur_t, err_msg=label)


@pytest.mark.parametrize("case", range(12))
def test_context_cache_matches_oracle_on_random_decode_loops(case):
    rng = np.random.default_rng(50260 + case)
    tokens, offsets = small_random_batch(rng)
    B = offsets.size - 1
    n_min = int(rng.integers(1, 5))
    n_max = int(rng.integers(n_min, 5))
    min_count = tuple(int(x) for x in rng.integers(1, 4, size=4))
    share = tuple((int(a), int(a) + int(c)) for a, c in zip(rng.integers(1, 3, size=4), rng.integers(0, 4, size=4)))
    K = int(rng.integers(1, 13))
    W = 9
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 4 * W, seed=case)
    t, b, n = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (st, base, length))
    capd = torch.from_numpy(cap).to(DEV)
    cc = pkg.ContextCache(st.shape[0], n_min, n_max, min_count=min_count, share=share)
    cc.build(t, b, n)
    cur_t, cur_o = tokens, offsets
    for step in range(3):
        d, ln = cc.draft(t, b, n, K)
        wd, wl = oracle.ctx_draft(cur_t, cur_o, K, n_min=n_min, n_max=n_max, min_count=min_count, share=share,
                                  threads=16)
        label = f"case {case} step {step}: B={B} n=[{n_min},{n_max}] K={K} {min_count} {share}"
        np.testing.assert_array_equal(ln.cpu().numpy(), wl, err_msg=f"{label}: len")
        np.testing.assert_array_equal(d.cpu().numpy(), wd, err_msg=f"{label}: draft")
        acc = np.minimum(np.minimum(rng.integers(0, K + 1, size=B), wl), W - 1)   # the row holds W tokens
        commit = rng.integers(-3, 50, size=(B, W)).astype(np.int32)
        for r in range(B):
            commit[r, :acc[r]] = wd[r, :acc[r]]
        ncommit = (acc + 1).astype(np.int32)
        status = cc.append(t, b, n, capd, torch.from_numpy(commit).to(DEV), torch.from_numpy(ncommit).to(DEV))
        assert (status.cpu().numpy() == 0).all(), label
        cur_t, cur_o = oracle.append(cur_t, cur_o, commit, ncommit)


@pytest.mark.parametrize("case", range(10))
def test_index_two_launch_loop_matches_oracle_on_random_decode_loops(case):
    """The decode loop on the index in two launches a step (lookup_index_draft_plan,
    then lookup_index_verify_append) on random batches, block shapes, thresholds,
    key widths (3 bits: most requests on the fallback) and greedy or sampled
    verification with the block's point masses, against the oracle's draft,
    schedule, fuse, verify and append over three steps."""
    rng = np.random.default_rng(50260 + case)
    tokens, offsets = small_random_batch(rng)
    B = offsets.size - 1
    min_m = int(rng.integers(1, 7))
    max_m = int(rng.integers(min_m, 33))
    H = int(rng.integers(1, 33))
    T = int(rng.integers(0, 65 - H))
    P = H + T
    agree_n = int(rng.integers(0, H + 1))
    kw = dict(replace_min=int(rng.integers(1, 13)), agree_min=int(rng.integers(1, 13)), agree_n=agree_n,
              tail_min=int(rng.integers(1, 13)), slack=int(rng.integers(0, 4)),
              enter_steps=int(rng.integers(1, 4)), sticky=int(rng.integers(0, 5)))
    hash_bits = int(rng.choice([64, 64, 3]))
    sampled = bool(rng.random() < 0.5)
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 4 * (P + 1), seed=case)
    t, b, n = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (st, base, length))
    capd = torch.from_numpy(cap).to(DEV)
    idx = pkg.NgramIndex(st.shape[0], min_m, max_m, hash_bits=hash_bits)
    idx.build(t, b, n)
    cur_t, cur_o = tokens, offsets
    st_o = np.zeros((B, 3), np.int32)
    st_g = torch.from_numpy(st_o.copy()).to(DEV)
    committed = np.full(B, H + 1, np.int32)
    label = f"case {case}: B={B} m=[{min_m},{max_m}] H={H} T={T} bits={hash_bits} sampled={sampled} {kw}"
    for step in range(3):
        d_o, l_o, p_o, m_o = oracle.lookup_draft(cur_t, cur_o, min_m, max_m, P, threads=16)
        md = rng.integers(-2, 4, size=(B, H)).astype(np.int32)
        take = rng.random(B) < 0.5
        md[take] = d_o[take, :H]
        lg_o = oracle.schedule(m_o, committed, st_o, H, T, tail_min=kw["tail_min"], slack=kw["slack"],
                               enter_steps=kw["enter_steps"], sticky=kw["sticky"])
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T, replace_min=kw["replace_min"],
                                         agree_min=kw["agree_min"], agree_n=agree_n, tail_min=kw["tail_min"])
        lg, blk, ln, pm, ml, dl, fb = idx.draft_plan(t, b, n, torch.from_numpy(md).to(DEV),
                                                     torch.from_numpy(committed).to(DEV), st_g, H, T, **kw)
        at = f"{label} step {step}"
        for name, g, w in (("long", lg, lg_o), ("block", blk, blk_o), ("len", ln, len_o), ("point mass", pm, pm_o),
                           ("mlen", ml, m_o), ("draft len", dl, l_o), ("state", st_g, st_o)):
            np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=f"{at}: {name}")
        target = rng.integers(-3, 50, size=(B, P + 1)).astype(np.int32)
        f = rng.integers(0, P + 1, size=B)
        for r in range(B):
            target[r, :f[r]] = blk_o[r, :f[r]]
        smp = {}
        if sampled:
            smp = dict(probs=rng.random((B, P), dtype=np.float32),
                       qprobs=(1.0 - rng.random((B, P), dtype=np.float32)).astype(np.float32),
                       u=rng.random((B, P), dtype=np.float32))
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target, point_mass=pm_o if sampled else None, **smp)
        acc, com, nc, status = idx.verify_append(blk, ln, torch.from_numpy(target).to(DEV), t, b, n, capd,
                                                 **({k: torch.from_numpy(v).to(DEV) for k, v in smp.items()}
                                                    | ({"point_mass": pm} if sampled else {})))
        for name, g, w in (("accepted", acc, acc_o), ("commit", com, com_o), ("ncommit", nc, nc_o)):
            np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=f"{at}: {name}")
        assert (status.cpu().numpy() == 0).all(), at
        cur_t, cur_o = oracle.append(cur_t, cur_o, com_o, nc_o)
        got_t, got_o = gen.csr_of_slabs(t.cpu().numpy(), base, n.cpu().numpy())
        np.testing.assert_array_equal(got_o, cur_o, err_msg=at)
        np.testing.assert_array_equal(got_t, cur_t, err_msg=at)
        committed = nc_o


@pytest.mark.parametrize("case", range(10))
def test_index_plain_lookup_loop_matches_oracle_on_random_batches(case):
    """Prompt-lookup decoding without a draft model through
    lookup_index_verify_append_draft: the block is the previous step's lookup
    draft, verified greedily (against a target that agrees on a random prefix)
    or by the sampled rule, then appended and drafted again, three steps, against
    the oracle's verify, append and draft.  Random batches, m ranges, K, key
    widths (3 bits: the exact scan), and one batch of more requests than a wave
    of append CTAs holds (the calls in order)."""
    rng = np.random.default_rng(60260 + case)
    if case == 9:                                        # more than one wave: many short requests
        lengths = rng.integers(0, 300, size=5000)
        tokens = rng.integers(0, 5, size=int(lengths.sum())).astype(np.int32)
        offsets = gen.offsets_from_lengths(lengths).astype(np.int64)
    else:
        tokens, offsets = small_random_batch(rng)
    B = offsets.size - 1
    min_m = int(rng.integers(1, 7))
    max_m = int(rng.integers(min_m, 33))
    K = int(rng.integers(1, 33))
    hash_bits = int(rng.choice([64, 64, 3]))
    sampled = bool(rng.random() < 0.5)
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 4 * (K + 1), seed=case)
    t, b, n = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (st, base, length))
    capd = torch.from_numpy(cap).to(DEV)
    idx = pkg.NgramIndex(st.shape[0], min_m, max_m, hash_bits=hash_bits)
    idx.build(t, b, n)
    cur_t, cur_o = tokens, offsets
    want = oracle.lookup_draft(cur_t, cur_o, min_m, max_m, K, threads=16)
    blk_o, len_o = want[0], want[1]
    blk_g, len_g = torch.from_numpy(blk_o).to(DEV), torch.from_numpy(len_o).to(DEV)
    label = f"case {case}: B={B} m=[{min_m},{max_m}] K={K} bits={hash_bits} sampled={sampled}"
    for step in range(3):
        target = rng.integers(-3, 50, size=(B, K + 1)).astype(np.int32)
        f = rng.integers(0, K + 1, size=B)
        for r in range(B):
            target[r, :f[r]] = blk_o[r, :f[r]]
        smp = {}
        if sampled:
            smp = dict(probs=rng.random((B, K), dtype=np.float32),
                       qprobs=(1.0 - rng.random((B, K), dtype=np.float32)).astype(np.float32),
                       u=rng.random((B, K), dtype=np.float32))
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target, **smp)
        cur_t, cur_o = oracle.append(cur_t, cur_o, com_o, nc_o)
        want = oracle.lookup_draft(cur_t, cur_o, min_m, max_m, K, threads=16)
        got = idx.verify_append_draft(blk_g, len_g, torch.from_numpy(target).to(DEV), t, b, n, capd, K,
                                      **{k: torch.from_numpy(v).to(DEV) for k, v in smp.items()})
        acc, com, nc, status, d, dl, pos, m, fb = got
        at = f"{label} step {step}"
        for name, g, w in (("accepted", acc, acc_o), ("commit", com, com_o), ("ncommit", nc, nc_o),
                           ("draft", d, want[0]), ("draft len", dl, want[1]), ("pos", pos, want[2]),
                           ("mlen", m, want[3])):
            np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=f"{at}: {name}")
        assert (status.cpu().numpy() == 0).all(), at
        blk_o, len_o = want[0], want[1]
        blk_g, len_g = d, dl
    got_t, got_o = gen.csr_of_slabs(t.cpu().numpy(), base, n.cpu().numpy())
    np.testing.assert_array_equal(got_o, cur_o, err_msg=label)
    np.testing.assert_array_equal(got_t, cur_t, err_msg=label)
