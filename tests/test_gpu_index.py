"""GPU parity of the incremental n-gram index (include/lookup_index.h).

The index must return exactly the oracle's draft (the definition of the draft
step) for the histories it holds: after a build, after every append of a
multi-step decode loop, with keys forced to share slots (the exact fallback),
and with a table too small to hold them.  Histories sit in capacity-padded
slabs with gaps (gen.slabs_from_batch); the oracle reads the same histories
as a CSR batch.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle

torch = pytest.importorskip("torch")
pkg = pytest.importorskip("prompt_lookup_speculative_gb300")

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def oracle_draft(slab_t, base, length, min_m, max_m, K):
    t, o = gen.csr_of_slabs(slab_t, base, length)
    return oracle.lookup_draft(t, o, min_m, max_m, K, threads=16)


def check_draft(got, want):
    d, ln, pos, m = (host(x) for x in got[:4])
    wd, wl, wp, wm = want
    np.testing.assert_array_equal(m, wm)
    np.testing.assert_array_equal(pos, wp)
    np.testing.assert_array_equal(ln, wl)
    np.testing.assert_array_equal(d, wd)


def built(slab_t, base, length, min_m, max_m, hash_bits=64, slots=None):
    t, b, n = dev(slab_t), dev(base), dev(length)
    idx = pkg.NgramIndex(slab_t.shape[0], min_m, max_m, hash_bits=hash_bits, slots=slots)
    idx.build(t, b, n)
    return idx, t, b, n


@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_index_draft_matches_oracle(name):
    w = gen.make_workload(name)
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 32, seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    got = idx.draft(t, b, n, w.K, with_fallback=True)
    check_draft(got, oracle_draft(st, base, length, w.min_m, w.max_m, w.K))
    assert host(got[4]).sum() == 0                      # 64-bit keys: no request needed the fallback


@pytest.mark.parametrize("min_m,max_m,K", [(1, 3, 5), (2, 8, 0), (4, 4, 64), (3, 32, 7), (1, 1, 1)])
def test_index_parameters_and_short_histories(min_m, max_m, K):
    rng = gen.rng_for(min_m * 100 + max_m, 31)
    lengths = [0, 1, 2, 3, 4, 5, 6, 7, 8, 12, 13, 33, 100, 700]
    hist = [rng.integers(0, 3, size=L).astype(np.int32) for L in lengths]
    tokens = np.concatenate(hist)
    offsets = gen.offsets_from_lengths(lengths)
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 16, seed=3)
    idx, t, b, n = built(st, base, length, min_m, max_m)
    check_draft(idx.draft(t, b, n, K), oracle_draft(st, base, length, min_m, max_m, K))


@pytest.mark.parametrize("hash_bits", [1, 3, 8, 14])
@pytest.mark.parametrize("name", ["tiny", "periodic"])
def test_shared_slots_fall_back_exactly(hash_bits, name):
    """With few key bits most keys share slots; the candidates that do not check
    out send their requests to the brute-force scan, and the result stays exact."""
    w = gen.make_workload(name)
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 0, seed=5)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m, hash_bits=hash_bits)
    got = idx.draft(t, b, n, w.K, with_fallback=True)
    check_draft(got, oracle_draft(st, base, length, w.min_m, w.max_m, w.K))
    if hash_bits <= 8:
        assert host(got[4]).sum() > 0


def test_overflowing_table_falls_back_exactly():
    w = gen.make_workload("tiny")
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 0, seed=6)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m, slots=1024)   # far too small
    got = idx.draft(t, b, n, w.K, with_fallback=True)
    check_draft(got, oracle_draft(st, base, length, w.min_m, w.max_m, w.K))
    assert host(got[4]).all()


@pytest.mark.parametrize("name", ["tiny", "recitation25k", "periodic", "chats"])
def test_index_decode_loop(name):
    """Draft from the index, commit a synthetic continuation (an accepted prefix
    of the draft and one more token), append it in place, and compare both the
    histories and the next draft with the oracle, for several steps."""
    w = gen.make_workload(name)
    W = 16
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 6 * W, seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    capd = dev(cap)
    B = w.B
    cur_t, cur_o = w.tokens, w.offsets
    rng = gen.rng_for(w.seed, 41)
    for step in range(6):
        got = idx.draft(t, b, n, w.K, with_fallback=True)
        want = oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, w.K, threads=16)
        check_draft(got, want)
        # commit: an accepted prefix of the draft (or of random tokens), then one more token
        acc = rng.integers(0, W, size=B)
        commit = rng.integers(0, 50, size=(B, W)).astype(np.int32)
        d = want[0]
        for r in range(B):
            k = min(int(acc[r]), w.K) if want[1][r] > 0 else 0
            commit[r, :k] = d[r, :k]
        ncommit = (np.minimum(acc, w.K) + 1).astype(np.int32)
        status = idx.append(t, b, n, capd, dev(commit), dev(ncommit))
        assert (host(status) == 0).all()
        cur_t, cur_o = oracle.append(cur_t, cur_o, commit, ncommit)
        got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
        np.testing.assert_array_equal(got_o, cur_o)
        np.testing.assert_array_equal(got_t, cur_t)


def test_append_status_full_slab_and_mismatch():
    w = gen.make_workload("tiny")
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 4, seed=8)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    commit = np.arange(8 * 6, dtype=np.int32).reshape(8, 6)
    ncommit = np.array([0, 4, 5, 6, 1, 2, 3, 4], np.int32)          # 5 and 6 do not fit in 4 spare slots
    status = host(idx.append(t, b, n, dev(cap), dev(commit), dev(ncommit)))
    assert list(status) == [0, 0, 1, 1, 0, 0, 0, 0]
    assert list(host(n)) == list(length + np.where(status == 0, ncommit, 0))
    # the index was built for min_m = 4: other parameters fail their requests
    status = host(pkg.lookup_index_append(t, b, n, dev(cap), dev(commit), dev(np.zeros(8, np.int32)), 3, 12,
                                          idx.memory, idx.slots))
    assert (status == 2).all()
    d, ln, pos, m = pkg.lookup_index_draft(t, b, n, 3, 12, 15, idx.memory, idx.slots)
    assert (host(ln) == pkg.LEN_FAILED).all()
    # and the right parameters still work on the appended histories
    t2, o2 = gen.csr_of_slabs(host(t), base, host(n))
    check_draft(idx.draft(t, b, n, 15), oracle.lookup_draft(t2, o2, 4, 12, 15))


@pytest.mark.parametrize("B", [300, 12000])
def test_append_both_launch_shapes(B):
    """The append runs one CTA per request when the batch fits in one wave of
    them, else dense tasks then a length pass.  Both must write the same tokens,
    lengths and statuses, and leave an index that drafts exactly."""
    rng = np.random.default_rng(B)
    lengths = rng.integers(0, 60, size=B)
    tokens = rng.integers(0, 6, size=int(lengths.sum())).astype(np.int32)
    offsets = gen.offsets_from_lengths(lengths)
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 4, seed=B)
    idx, t, b, n = built(st, base, length, 4, 12)
    W = 6
    commit = rng.integers(0, 6, size=(B, W)).astype(np.int32)
    ncommit = rng.integers(0, W + 1, size=B).astype(np.int32)       # 5 and 6 do not fit in 4 spare slots
    status = host(idx.append(t, b, n, dev(cap), dev(commit), dev(ncommit)))
    fits = ncommit <= 4
    np.testing.assert_array_equal(status, np.where(fits, 0, 1))
    np.testing.assert_array_equal(host(n), length + np.where(fits, ncommit, 0))
    want_t, want_o = oracle.append(tokens, offsets, commit, np.where(fits, ncommit, 0).astype(np.int32))
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_o, want_o)
    np.testing.assert_array_equal(got_t, want_t)
    check_draft(idx.draft(t, b, n, 7), oracle.lookup_draft(want_t, want_o, 4, 12, 7, threads=16))


def test_index_agrees_with_the_scan():
    """The index and the scan kernel give the same drafts on the same histories."""
    w = gen.make_workload("ragged262k")
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 0, seed=9)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    a = idx.draft(t, b, n, w.K)
    s = pkg.lookup_draft_ex(dev(w.tokens), dev(w.offsets), w.min_m, w.max_m, w.K)
    for x, y in zip(a, s):
        np.testing.assert_array_equal(host(x), host(y))


@pytest.mark.parametrize("period", [1, 2, 3, 5])
def test_append_repeated_ngrams_in_one_call(period):
    """Commits that repeat their own n-grams: several threads of one append
    update the same slots at once (the contended path of the slot update)."""
    rng = gen.rng_for(period, 51)
    B, W = 24, 32
    lengths = rng.integers(0, 300, size=B)
    tokens = rng.integers(0, 20, size=int(lengths.sum())).astype(np.int32)
    offsets = gen.offsets_from_lengths(lengths)
    st, base, length, cap = gen.slabs_from_batch(tokens, offsets, 4 * W, seed=period)
    idx, t, b, n = built(st, base, length, 4, 12)
    cur_t, cur_o = tokens, offsets
    for step in range(3):
        pattern = rng.integers(0, 20, size=(B, period)).astype(np.int32)
        commit = np.tile(pattern, (1, W // period + 1))[:, :W].astype(np.int32)
        ncommit = rng.integers(W // 2, W + 1, size=B).astype(np.int32)
        assert (host(idx.append(t, b, n, dev(cap), dev(commit), dev(ncommit))) == 0).all()
        cur_t, cur_o = oracle.append(cur_t, cur_o, commit, ncommit)
        got = idx.draft(t, b, n, 15, with_fallback=True)
        check_draft(got, oracle.lookup_draft(cur_t, cur_o, 4, 12, 15))
        assert host(got[4]).sum() == 0


# ---------------------------------------------------- index draft, then plan ----
def _plan_inputs(B, H, T, d_o, seed):
    rng = gen.rng_for(seed, 43)
    md = rng.integers(0, 50, size=(B, H)).astype(np.int32)
    take = rng.random(B) < 0.4
    md[take] = d_o[take, :H]
    committed = rng.integers(1, H + T + 2, size=B).astype(np.int32)
    state = np.stack([rng.integers(0, 2, B), rng.integers(0, 3, B), rng.integers(0, 4, B)], 1).astype(np.int32)
    return md, committed, state


def _oracle_plan(d_o, m_o, md, committed, state, H, T):
    st = state.copy()
    lg = oracle.schedule(m_o, committed, st, H, T)
    blk, ln, pm = oracle.fuse(d_o, m_o, md, lg, H, T)
    return lg, blk, ln, pm, st


@pytest.mark.parametrize("hash_bits", [64, 3])
@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_index_draft_plan_is_index_draft_then_plan(name, hash_bits):
    """hash_bits = 3: nearly all keys share slots, so most requests take the
    brute-force path, and the plan must follow its draft as well."""
    w = gen.make_workload(name)
    H, T = 7, 8
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 32, seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m, hash_bits=hash_bits)
    d_o, l_o, p_o, m_o = oracle_draft(st, base, length, w.min_m, w.max_m, H + T)
    md, committed, state = _plan_inputs(w.B, H, T, d_o, w.seed)
    lg_o, blk_o, len_o, pm_o, st_o = _oracle_plan(d_o, m_o, md, committed, state, H, T)
    st_g = dev(state)
    lg, blk, ln, pm, ml, dl, fb = idx.draft_plan(t, b, n, dev(md), dev(committed), st_g, H, T)
    for nm, g, e in (("long", lg, lg_o), ("block", blk, blk_o), ("len", ln, len_o), ("point mass", pm, pm_o),
                     ("mlen", ml, m_o), ("draft len", dl, l_o), ("state", st_g, st_o)):
        np.testing.assert_array_equal(host(g), e, err_msg=nm)
    if hash_bits == 64:
        assert host(fb).sum() == 0


@pytest.mark.parametrize("name", ["recitation25k", "chats"])
def test_index_decode_loop_with_plan(name):
    """Index draft + plan -> greedy verify -> index append, four steps, against the
    oracle's draft -> schedule -> fuse -> verify -> append."""
    w = gen.make_workload(name)
    H, T = 7, 8
    W = H + T + 1
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 5 * W, seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    capd = dev(cap)
    B = w.B
    cur_t, cur_o = w.tokens, w.offsets
    st_o = np.zeros((B, 3), np.int32)
    st_g = dev(st_o)
    committed = np.full(B, H + 1, np.int32)
    for step in range(4):
        d_o, l_o, p_o, m_o = oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, H + T, threads=16)
        md, _, _ = _plan_inputs(B, H, T, d_o, step)
        lg_o = oracle.schedule(m_o, committed, st_o, H, T)
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T)
        lg, blk, ln, pm, ml, dl, fb = idx.draft_plan(t, b, n, dev(md), dev(committed), st_g, H, T)
        for nm, g, e in (("long", lg, lg_o), ("block", blk, blk_o), ("len", ln, len_o), ("state", st_g, st_o)):
            np.testing.assert_array_equal(host(g), e, err_msg=f"{nm}, step {step}")
        rng = gen.rng_for(step, 44)
        target = rng.integers(0, 50, size=(B, H + T + 1)).astype(np.int32)
        f = rng.integers(0, H + T + 1, size=B)
        for r in range(B):
            target[r, :f[r]] = blk_o[r, :f[r]]
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target)
        assert (host(idx.append(t, b, n, capd, dev(com_o), dev(nc_o))) == 0).all()
        cur_t, cur_o = oracle.append(cur_t, cur_o, com_o, nc_o)
        committed = nc_o


# --------------------------------------------------- verify, then append ----
def _verify_inputs(B, P, seed, mode):
    blk, ln, tg, pr, qp, pm, u = gen.loop_verify_inputs(B, P, seed)
    if mode == "greedy":
        return (blk, ln, tg), {}
    return (blk, ln, tg), dict(probs=pr, qprobs=qp, point_mass=pm, u=u)


@pytest.mark.parametrize("mode", ["greedy", "sampled"])
@pytest.mark.parametrize("name", ["tiny", "recitation25k", "chats"])
def test_index_verify_append_is_verify_then_append(name, mode):
    """recitation25k and tiny: one launch (a CTA per request verifies, then
    appends); chats (4,096 requests, more than one wave): the two calls."""
    w = gen.make_workload(name)
    P = 15
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 3 * (P + 1), seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    (blk, ln, tg), smp = _verify_inputs(w.B, P, w.seed, mode)
    acc_o, com_o, nc_o = oracle.verify(blk, ln, tg, **smp)
    acc, com, nc, status = idx.verify_append(dev(blk), dev(ln), dev(tg), t, b, n, dev(cap),
                                             **{k: dev(v) for k, v in smp.items()})
    for nm, g, e in (("accepted", acc, acc_o), ("commit", com, com_o), ("ncommit", nc, nc_o)):
        np.testing.assert_array_equal(host(g), e, err_msg=nm)
    assert (host(status) == 0).all()
    cur_t, cur_o = oracle.append(w.tokens, w.offsets, com_o, nc_o)
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_o, cur_o)
    np.testing.assert_array_equal(got_t, cur_t)
    check_draft(idx.draft(t, b, n, w.K), oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, w.K, threads=16))


def test_index_verify_append_error_rows_and_full_slabs():
    """A block length outside [0, P] gives the header's error row (accepted -1, no
    committed token, commit row -1) and appends nothing; a request whose slab
    cannot hold its committed tokens gets status 1 and keeps its history, while
    its verification outputs are still written."""
    w = gen.make_workload("recitation25k")
    P = 15
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, P + 1, seed=w.seed)
    cap = cap.copy()
    (blk, ln, tg), _ = _verify_inputs(w.B, P, 7, "greedy")
    bad = np.zeros(w.B, bool)
    bad[[3, 17]] = True
    ln_bad = ln.copy()
    ln_bad[3], ln_bad[17] = -1, P + 4
    full = np.zeros(w.B, bool)
    full[[5, 40]] = True
    cap[full] = length[full]                              # no room at all: any commit overflows
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    ok = ~bad
    acc_o, com_o, nc_o = oracle.verify(blk[ok], ln[ok], tg[ok])
    acc, com, nc, status = idx.verify_append(dev(blk), dev(ln_bad), dev(tg), t, b, n, dev(cap))
    acc, com, nc, status = host(acc), host(com), host(nc), host(status)
    np.testing.assert_array_equal(acc[ok], acc_o)
    np.testing.assert_array_equal(com[ok], com_o)
    np.testing.assert_array_equal(nc[ok], nc_o)
    assert (acc[bad] == -1).all() and (nc[bad] == 0).all() and (com[bad] == -1).all()
    want_status = np.where(full & ok, 1, 0)
    np.testing.assert_array_equal(status, want_status)
    nc_eff = np.zeros(w.B, np.int32)
    nc_eff[ok] = nc_o
    nc_eff[full] = 0
    com_eff = np.full((w.B, P + 1), -1, np.int32)
    com_eff[ok] = com_o
    cur_t, cur_o = oracle.append(w.tokens, w.offsets, com_eff, nc_eff)
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_o, cur_o)
    np.testing.assert_array_equal(got_t, cur_t)
    check_draft(idx.draft(t, b, n, w.K), oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, w.K, threads=16))


@pytest.mark.parametrize("name", ["recitation25k", "periodic"])
def test_index_decode_loop_in_two_launches(name):
    """The decode loop on the index with lookup_index_draft_plan and
    lookup_index_verify_append (two launches a step), four steps, against the
    oracle's draft -> schedule -> fuse -> verify -> append."""
    w = gen.make_workload(name)
    H, T = 7, 8
    P = H + T
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 5 * (P + 1), seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    capd = dev(cap)
    B = w.B
    cur_t, cur_o = w.tokens, w.offsets
    st_o = np.zeros((B, 3), np.int32)
    st_g = dev(st_o)
    committed = np.full(B, H + 1, np.int32)
    for step in range(4):
        d_o, l_o, p_o, m_o = oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, P, threads=16)
        md, _, _ = _plan_inputs(B, H, T, d_o, step)
        lg_o = oracle.schedule(m_o, committed, st_o, H, T)
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T)
        lg, blk, ln, pm, ml, dl, fb = idx.draft_plan(t, b, n, dev(md), dev(committed), st_g, H, T)
        np.testing.assert_array_equal(host(blk), blk_o, err_msg=f"block, step {step}")
        np.testing.assert_array_equal(host(ln), len_o, err_msg=f"len, step {step}")
        rng = gen.rng_for(step, 45)
        target = rng.integers(0, 50, size=(B, P + 1)).astype(np.int32)
        f = rng.integers(0, P + 1, size=B)
        for r in range(B):
            target[r, :f[r]] = blk_o[r, :f[r]]
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target)
        acc, com, nc, status = idx.verify_append(blk, ln, dev(target), t, b, n, capd)
        np.testing.assert_array_equal(host(nc), nc_o, err_msg=f"ncommit, step {step}")
        np.testing.assert_array_equal(host(com), com_o, err_msg=f"commit, step {step}")
        assert (host(status) == 0).all()
        cur_t, cur_o = oracle.append(cur_t, cur_o, com_o, nc_o)
        committed = nc_o
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_t, cur_t)
    np.testing.assert_array_equal(got_o, cur_o)


def test_index_verify_append_with_empty_blocks():
    """P = 0: no proposals (the block pointer may be NULL); every request commits
    the target's one token, which the append writes and indexes."""
    w = gen.make_workload("periodic")
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 8, seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    blk = np.zeros((w.B, 0), np.int32)
    ln = np.zeros(w.B, np.int32)
    tg = gen.rng_for(5, 46).integers(0, 50, size=(w.B, 1)).astype(np.int32)
    acc_o, com_o, nc_o = oracle.verify(blk, ln, tg)
    lib = pkg.load_library()
    acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    com = torch.empty((w.B, 1), dtype=torch.int32, device="cuda")
    nc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    status = torch.empty(w.B, dtype=torch.int32, device="cuda")
    lnd, tgd, capd = dev(ln), dev(tg), dev(cap)
    rc = lib.lookup_index_verify_append(None, lnd.data_ptr(), tgd.data_ptr(), None, None, None, None, w.B, 0,
                                        t.data_ptr(), b.data_ptr(), n.data_ptr(), capd.data_ptr(), w.min_m, w.max_m,
                                        idx.memory.data_ptr(), idx.slots, 64, acc.data_ptr(), com.data_ptr(),
                                        nc.data_ptr(), status.data_ptr(), None)
    assert rc == 0
    np.testing.assert_array_equal(host(acc), acc_o)
    np.testing.assert_array_equal(host(com), com_o)
    np.testing.assert_array_equal(host(nc), nc_o)
    assert (host(status) == 0).all()
    cur_t, cur_o = oracle.append(w.tokens, w.offsets, com_o, nc_o)
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_t, cur_t)
    check_draft(idx.draft(t, b, n, w.K), oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, w.K, threads=16))


# ------------------------------------------- verify, append, then draft ----
@pytest.mark.parametrize("mode", ["greedy", "sampled"])
@pytest.mark.parametrize("name,hash_bits", [("tiny", 64), ("recitation25k", 64), ("recitation25k", 3), ("chats", 64)])
def test_index_verify_append_draft_is_the_composition(name, hash_bits, mode):
    """One launch on one-wave batches (a CTA per request verifies, appends and
    drafts), the calls on chats; with 3-bit keys most requests draft through the
    exact scan.  Against the oracle's verify, append and draft."""
    w = gen.make_workload(name)
    P = 15
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 3 * (P + 1), seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m, hash_bits=hash_bits)
    (blk, ln, tg), smp = _verify_inputs(w.B, P, w.seed + 1, mode)
    acc_o, com_o, nc_o = oracle.verify(blk, ln, tg, **smp)
    cur_t, cur_o = oracle.append(w.tokens, w.offsets, com_o, nc_o)
    want = oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, w.K, threads=16)
    got = idx.verify_append_draft(dev(blk), dev(ln), dev(tg), t, b, n, dev(cap), w.K,
                                  **{k: dev(v) for k, v in smp.items()})
    acc, com, nc, status, d, dl, pos, m, fb = got
    for nm, g, e in (("accepted", acc, acc_o), ("commit", com, com_o), ("ncommit", nc, nc_o)):
        np.testing.assert_array_equal(host(g), e, err_msg=nm)
    assert (host(status) == 0).all()
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_t, cur_t)
    check_draft((d, dl, pos, m), want)
    if hash_bits == 64:
        assert host(fb).sum() == 0


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("name", ["recitation25k", "periodic", "tiny"])
def test_index_plain_lookup_decode_loop_in_one_launch(name, in_place):
    """Prompt-lookup decoding without a draft model: the block is the previous
    step's lookup draft (K = P proposals, or none without a match), the target
    agrees with it on a random prefix, and each step is one call of
    lookup_index_verify_append_draft; in_place: the draft overwrites the block
    and its lengths.  Five steps against the oracle."""
    w = gen.make_workload(name)
    P = 15
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, 6 * (P + 1), seed=w.seed)
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    capd = dev(cap)
    cur_t, cur_o = w.tokens, w.offsets
    want = oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, P, threads=16)
    blk_o, len_o = want[0], want[1]
    blk_g, len_g = dev(blk_o), dev(len_o)
    for step in range(5):
        rng = gen.rng_for(step, 47)
        target = rng.integers(0, 50, size=(w.B, P + 1)).astype(np.int32)
        f = rng.integers(0, P + 1, size=w.B)
        for r in range(w.B):
            target[r, :f[r]] = blk_o[r, :f[r]]
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target)
        cur_t, cur_o = oracle.append(cur_t, cur_o, com_o, nc_o)
        want = oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, P, threads=16)
        if in_place:
            outs = (torch.empty(w.B, dtype=torch.int32, device="cuda"),
                    torch.empty((w.B, P + 1), dtype=torch.int32, device="cuda"),
                    torch.empty(w.B, dtype=torch.int32, device="cuda"),
                    torch.empty(w.B, dtype=torch.int32, device="cuda"), blk_g, len_g,
                    torch.empty(w.B, dtype=torch.int32, device="cuda"),
                    torch.empty(w.B, dtype=torch.int32, device="cuda"),
                    torch.empty(w.B, dtype=torch.int32, device="cuda"))
            got = pkg.lookup_index_verify_append_draft(blk_g, len_g, dev(target), t, b, n, capd, w.min_m, w.max_m,
                                                       idx.memory, idx.slots, P, out=outs)
        else:
            got = idx.verify_append_draft(blk_g, len_g, dev(target), t, b, n, capd, P)
        acc, com, nc, status, d, dl, pos, m, fb = got
        np.testing.assert_array_equal(host(nc), nc_o, err_msg=f"ncommit, step {step}")
        np.testing.assert_array_equal(host(com), com_o, err_msg=f"commit, step {step}")
        assert (host(status) == 0).all()
        check_draft((d, dl, pos, m), want)
        blk_o, len_o = want[0], want[1]
        blk_g, len_g = d, dl
    got_t, got_o = gen.csr_of_slabs(host(t), base, host(n))
    np.testing.assert_array_equal(got_t, cur_t)


def test_index_verify_append_draft_error_rows_and_full_slabs():
    """As for verify-and-append: an out-of-range block length gives the error row
    and appends nothing, a full slab gets status 1 and keeps its history; every
    request is then drafted from its history as it stands."""
    w = gen.make_workload("recitation25k")
    P = 15
    st, base, length, cap = gen.slabs_from_batch(w.tokens, w.offsets, P + 1, seed=w.seed)
    cap = cap.copy()
    (blk, ln, tg), _ = _verify_inputs(w.B, P, 9, "greedy")
    bad = np.zeros(w.B, bool)
    bad[[2, 30]] = True
    ln_bad = ln.copy()
    ln_bad[2], ln_bad[30] = -3, P + 1
    full = np.zeros(w.B, bool)
    full[[7, 41]] = True
    cap[full] = length[full]
    idx, t, b, n = built(st, base, length, w.min_m, w.max_m)
    ok = ~bad
    acc_o, com_o, nc_o = oracle.verify(blk[ok], ln[ok], tg[ok])
    got = idx.verify_append_draft(dev(blk), dev(ln_bad), dev(tg), t, b, n, dev(cap), w.K)
    acc, com, nc, status, d, dl, pos, m, fb = (host(x) for x in got)
    np.testing.assert_array_equal(acc[ok], acc_o)
    np.testing.assert_array_equal(nc[ok], nc_o)
    assert (acc[bad] == -1).all() and (nc[bad] == 0).all()
    np.testing.assert_array_equal(status, np.where(full & ok, 1, 0))
    nc_eff = np.zeros(w.B, np.int32)
    nc_eff[ok] = nc_o
    nc_eff[full] = 0
    com_eff = np.full((w.B, P + 1), -1, np.int32)
    com_eff[ok] = com_o
    cur_t, cur_o = oracle.append(w.tokens, w.offsets, com_eff, nc_eff)
    want = oracle.lookup_draft(cur_t, cur_o, w.min_m, w.max_m, w.K, threads=16)
    for nm, g, e in (("draft", d, want[0]), ("draft len", dl, want[1]), ("pos", pos, want[2]), ("mlen", m, want[3])):
        np.testing.assert_array_equal(g, e, err_msg=nm)
