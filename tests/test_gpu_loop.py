"""GPU parity of the decode-loop steps (include/lookup_loop.h) against the oracle.

Every comparison is element by element and exact: the steps are integer work,
and the one floating-point decision (the sampled acceptance test u * q < p) is
taken in float32 on both sides, as the header states.  Inputs come from the
seeded generators in gen/, at sizes the oracle finishes in well under a second,
and at the full sizes of the drafting workloads for the append.
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
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


# ------------------------------------------------------------------ fusion ----
@pytest.mark.parametrize("B", [1, 7, 4096])
@pytest.mark.parametrize("H,T,agree_n", [(7, 8, 2), (3, 2, 0), (3, 2, 3), (1, 0, 1), (7, 0, 2), (16, 48, 2)])
@pytest.mark.parametrize("seed", [1, 2])
def test_fuse_matches_oracle(B, H, T, agree_n, seed):
    K = max(H + T, 15)
    ld, m, md, lg = gen.loop_fuse_inputs(B, K, H, T, agree_n, seed)
    want = oracle.fuse(ld, m, md, lg, H, T, agree_n=agree_n)
    got = pkg.lookup_fuse(dev(ld), dev(m), dev(md), dev(lg), H, T, agree_n=agree_n)
    for w, g in zip(want, got):
        np.testing.assert_array_equal(host(g), w)


@pytest.mark.parametrize("rm,am,tm", [(8, 6, 4), (4, 4, 4), (1, 20, 0), (13, 13, 13)])
def test_fuse_thresholds_and_no_long_flags(rm, am, tm):
    B, H, T = 2048, 7, 8
    ld, m, md, lg = gen.loop_fuse_inputs(B, 15, H, T, 2, 7)
    for long_block in (lg, None):
        want = oracle.fuse(ld, m, md, long_block, H, T, replace_min=rm, agree_min=am, tail_min=tm)
        got = pkg.lookup_fuse(dev(ld), dev(m), dev(md), dev(long_block), H, T, replace_min=rm,
                              agree_min=am, tail_min=tm)
        for w, g in zip(want, got):
            np.testing.assert_array_equal(host(g), w)


# -------------------------------------------------------------- scheduling ----
@pytest.mark.parametrize("B,steps", [(1, 64), (33, 40), (4096, 24)])
@pytest.mark.parametrize("params", [dict(), dict(slack=0, enter_steps=1, sticky=0),
                                    dict(slack=3, enter_steps=3, sticky=5, tail_min=6)])
def test_schedule_trace_matches_oracle(B, steps, params):
    H, T = 7, 8
    mlen, committed = gen.loop_schedule_trace(B, steps, H, T, seed=B + steps)
    st_o = np.zeros((B, 3), np.int32)
    st_g = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    entered = 0
    for s in range(steps):
        want = oracle.schedule(mlen[s], committed[s], st_o, H, T, **params)
        got = pkg.lookup_schedule(dev(mlen[s]), dev(committed[s]), st_g, H, T, **params)
        np.testing.assert_array_equal(host(got), want, err_msg=f"step {s}")
        np.testing.assert_array_equal(host(st_g), st_o, err_msg=f"state after step {s}")
        entered += int(want.sum())
    if B > 1:
        assert 0 < entered < B * steps          # the trace really switches modes


# ------------------------------------------------------------ verification ----
@pytest.mark.parametrize("B", [1, 5, 4096])
@pytest.mark.parametrize("P", [0, 1, 15, 31, 32, 33, 70])
def test_verify_greedy_matches_oracle(B, P):
    block, ln, target, *_ = gen.loop_verify_inputs(B, P, seed=P + 11)
    want = oracle.verify(block, ln, target)
    got = pkg.lookup_verify(dev(block), dev(ln), dev(target))
    for w, g in zip(want, got):
        np.testing.assert_array_equal(host(g), w)


@pytest.mark.parametrize("B", [3, 4096])
@pytest.mark.parametrize("P", [1, 15, 40])
@pytest.mark.parametrize("with_q,with_pm", [(True, True), (True, False), (False, False), (False, True)])
def test_verify_sampled_matches_oracle(B, P, with_q, with_pm):
    block, ln, target, p, q, pm, u = gen.loop_verify_inputs(B, P, seed=P + 23)
    q = q if with_q else None
    pm = pm if with_pm else None
    want = oracle.verify(block, ln, target, probs=p, qprobs=q, point_mass=pm, u=u)
    got = pkg.lookup_verify(dev(block), dev(ln), dev(target), probs=dev(p), qprobs=dev(q),
                            point_mass=dev(pm), u=dev(u))
    for w, g in zip(want, got):
        np.testing.assert_array_equal(host(g), w)
    acc = want[0]
    assert 0 < (acc < ln).sum() < B or B < 10         # both full and partial acceptances occur


def test_verify_ties_reject():
    # u * q == p exactly is a rejection on both sides (strict comparison).
    P = 4
    block = np.array([[1, 2, 3, 4]], np.int32)
    target = np.array([[1, 2, 3, 4, 5]], np.int32)
    u = np.array([[0.25, 0.5, 0.75, 0.125]], np.float32)
    q = np.array([[1.0, 0.5, 1.0, 1.0]], np.float32)
    p = np.array([[0.5, 0.25, 0.9, 0.9]], np.float32)     # 0.5*0.5 == 0.25: reject at 1
    got = pkg.lookup_verify(dev(block), dev(np.array([P], np.int32)), dev(target), probs=dev(p),
                            qprobs=dev(q), u=dev(u))
    want = oracle.verify(block, [P], target, probs=p, qprobs=q, u=u)
    assert int(want[0][0]) == 1
    for w, g in zip(want, got):
        np.testing.assert_array_equal(host(g), w)


def test_verify_invalid_length_gives_error_row():
    block = np.arange(12, dtype=np.int32).reshape(3, 4)
    target = np.arange(15, dtype=np.int32).reshape(3, 5)
    ln = np.array([4, 5, -1], np.int32)                   # rows 1 and 2 are invalid
    acc, commit, nc = pkg.lookup_verify(dev(block), dev(ln), dev(target))
    acc, commit, nc = host(acc), host(commit), host(nc)
    assert list(acc[1:]) == [-1, -1] and list(nc[1:]) == [0, 0]
    assert (commit[1:] == -1).all()
    want = oracle.verify(block[:1], ln[:1], target[:1])  # the valid row is untouched by the others
    assert acc[0] == want[0][0] and list(commit[0]) == list(want[1][0])


# ------------------------------------------------------------------ append ----
def _append_case(tokens, offsets, W, seed, lead=0, unaligned=False):
    B = offsets.shape[0] - 1
    commit, ncommit = gen.loop_append_inputs(B, W, seed)
    if lead:
        tokens = np.concatenate([np.full(lead, -7, np.int32), tokens])
        offsets = offsets + lead
    want_t, want_o = oracle.append(tokens, offsets, commit, ncommit)
    t, o = dev(tokens), dev(offsets)
    cap = tokens.shape[0] + B * W + 8
    buf = torch.full((cap,), -99, dtype=torch.int32, device="cuda")
    out_t = buf[1:] if unaligned else buf[:-1]
    out_o = torch.empty(B + 1, dtype=torch.int64, device="cuda")
    pkg.lookup_append(t, o, dev(commit), dev(ncommit), out=(out_t, out_o))
    got_o = host(out_o)
    np.testing.assert_array_equal(got_o, want_o)
    got_t = host(out_t)
    np.testing.assert_array_equal(got_t[:want_t.shape[0]], want_t)
    assert (got_t[want_t.shape[0]:] == -99).all()          # nothing written past the batch


@pytest.mark.parametrize("lengths", [[0], [1], [5, 0, 0, 3], [0] * 100, [3000, 1, 0, 7777, 31],
                                     [127, 128, 129, 0, 256, 1, 1000], [511, 512, 513, 0, 1024, 2047, 1]])
@pytest.mark.parametrize("W", [0, 1, 16])
@pytest.mark.parametrize("lead,unaligned", [(5, False), (5, True), (0, True), (1, False), (2, True), (3, False)])
def test_append_small_and_ragged(lengths, W, lead, unaligned):
    rng = gen.rng_for(len(lengths) * 31 + W, 9)
    tokens = rng.integers(0, 1000, size=sum(lengths)).astype(np.int32)
    _append_case(tokens, gen.offsets_from_lengths(lengths), W, seed=W + 1, lead=lead, unaligned=unaligned)


@pytest.mark.parametrize("seed", range(6))
def test_append_random_batches(seed):
    rng = gen.rng_for(seed, 19)
    B = int(rng.integers(1, 3000))
    lengths = np.where(rng.random(B) < 0.2, 0, rng.integers(1, 2000, size=B))
    tokens = rng.integers(0, 1 << 30, size=int(lengths.sum())).astype(np.int32)
    _append_case(tokens, gen.offsets_from_lengths(lengths), int(rng.integers(1, 40)), seed=seed,
                 lead=int(rng.integers(0, 8)), unaligned=bool(seed % 2))


def test_append_clamps_counts():
    # counts outside [0, W] are clamped (the header's rule); the oracle takes the clamped counts
    rng = gen.rng_for(5, 21)
    lengths = [300, 0, 17, 129]
    tokens = rng.integers(0, 1000, size=sum(lengths)).astype(np.int32)
    offsets = gen.offsets_from_lengths(lengths)
    W = 4
    commit = rng.integers(0, 1000, size=(4, W)).astype(np.int32)
    ncommit = np.array([-3, 9, 4, 0], np.int32)
    want_t, want_o = oracle.append(tokens, offsets, commit, np.clip(ncommit, 0, W))
    out_t, out_o = pkg.lookup_append(dev(tokens), dev(offsets), dev(commit), dev(ncommit))
    np.testing.assert_array_equal(host(out_o), want_o)
    np.testing.assert_array_equal(host(out_t)[:want_t.shape[0]], want_t)


@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_append_full_workloads(name):
    w = gen.make_workload(name)
    _append_case(w.tokens, w.offsets, 16, seed=3)


def test_append_empty_batch():
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    o = torch.zeros(1, dtype=torch.int64, device="cuda")
    out_t, out_o = pkg.lookup_append(t, o, torch.zeros((0, 16), dtype=torch.int32, device="cuda"),
                                     torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert list(host(out_o)) == [0]


# ------------------------------------------------------------- whole loop ----
@pytest.mark.parametrize("name", ["tiny", "chats"])
def test_decode_loop_matches_oracle(name):
    """Draft -> fuse -> verify -> append -> schedule, several steps, both sides.

    The target model is synthetic: at each step the target tokens agree with
    the (already compared) proposal block on a random prefix, drawn on the host
    from the step's seed.  Every intermediate is compared exactly."""
    w = gen.make_workload(name)
    B, H, T = w.B, 7, 8
    K = H + T
    P = H + T
    tokens_o, offsets_o = w.tokens, w.offsets
    tokens_g, offsets_g = dev(w.tokens), dev(w.offsets)
    st_o = np.zeros((B, 3), np.int32)
    st_g = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    long_o = np.zeros(B, np.int32)
    long_g = torch.zeros(B, dtype=torch.int32, device="cuda")
    committed = np.full(B, H + 1, np.int32)
    for step in range(4):
        d_o, l_o, p_o, m_o = oracle.lookup_draft(tokens_o, offsets_o, w.min_m, w.max_m, K, threads=8)
        d_g, l_g, p_g, m_g = pkg.lookup_draft_ex(tokens_g, offsets_g, w.min_m, w.max_m, K)
        np.testing.assert_array_equal(host(d_g), d_o)
        np.testing.assert_array_equal(host(m_g), m_o)
        # scheduling from this step's match and the previous step's commit count
        lg_o = oracle.schedule(m_o, committed, st_o, H, T)
        pkg.lookup_schedule(m_g, dev(committed), st_g, H, T, out=long_g)
        np.testing.assert_array_equal(host(long_g), lg_o)
        # a synthetic draft model: the lookup head for a third of the requests
        rng = gen.rng_for(step, 77)
        md = rng.integers(0, 50, size=(B, H), dtype=np.int64).astype(np.int32)
        pick = rng.random(B) < 0.33
        md[pick] = d_o[pick, :H]
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T)
        blk_g, len_g, pm_g = pkg.lookup_fuse(d_g, m_g, dev(md), long_g, H, T)
        for a, b in ((blk_o, blk_g), (len_o, len_g), (pm_o, pm_g)):
            np.testing.assert_array_equal(host(b), a)
        # synthetic target: agree with the block on a random prefix
        target = rng.integers(0, 50, size=(B, P + 1), dtype=np.int64).astype(np.int32)
        f = rng.integers(0, P + 1, size=B)
        for r in range(B):
            target[r, :f[r]] = blk_o[r, :f[r]]
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target)
        acc_g, com_g, nc_g = pkg.lookup_verify(blk_g, len_g, dev(target))
        for a, b in ((acc_o, acc_g), (com_o, com_g), (nc_o, nc_g)):
            np.testing.assert_array_equal(host(b), a)
        tokens_o, offsets_o = oracle.append(tokens_o, offsets_o, com_o, nc_o)
        tokens_g, offsets_g = pkg.lookup_append(tokens_g, offsets_g, com_g, nc_g)
        np.testing.assert_array_equal(host(offsets_g), offsets_o)
        np.testing.assert_array_equal(host(tokens_g)[:offsets_o[-1]], tokens_o)
        committed = nc_o


@pytest.mark.parametrize("name,B_sub", [("tiny", None), ("chats", 1000), ("chats", None)])
def test_decode_loop_back_to_back(name, B_sub):
    """The same loop with no host synchronisation inside it: every kernel runs
    behind the previous one on the stream (programmatic dependent launch), the
    synthetic model and target are formed on the device with torch, and only the
    final histories and the last draft are compared with the oracle's loop.
    Batches of at most 1024 requests take the append that forms the new offsets
    itself, right behind the verify step that writes the counts."""
    w = gen.make_workload(name)
    tokens, offsets = w.tokens, w.offsets
    if B_sub is not None:
        offsets = offsets[:B_sub + 1]
        tokens = tokens[:offsets[-1]]
    B, H, T = offsets.shape[0] - 1, 7, 8
    K = P = H + T
    steps = 4
    rng = gen.rng_for(B, 78)
    md_rand = rng.integers(0, 50, size=(steps, B, H), dtype=np.int64).astype(np.int32)
    pick = rng.random((steps, B)) < 0.33
    tgt_rand = rng.integers(0, 50, size=(steps, B, P + 1), dtype=np.int64).astype(np.int32)
    f = rng.integers(0, P + 1, size=(steps, B))
    # the oracle's loop
    t_o, o_o = tokens, offsets
    st_o = np.zeros((B, 3), np.int32)
    committed = np.full(B, H + 1, np.int32)
    for s in range(steps):
        d_o, l_o, p_o, m_o = oracle.lookup_draft(t_o, o_o, w.min_m, w.max_m, K, threads=8)
        lg_o = oracle.schedule(m_o, committed, st_o, H, T)
        md = md_rand[s].copy()
        md[pick[s]] = d_o[pick[s], :H]
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T)
        target = tgt_rand[s].copy()
        for r in range(B):
            target[r, :f[s, r]] = blk_o[r, :f[s, r]]
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target)
        t_o, o_o = oracle.append(t_o, o_o, com_o, nc_o)
        committed = nc_o
    d_last, _, _, m_last = oracle.lookup_draft(t_o, o_o, w.min_m, w.max_m, K, threads=8)
    # the device's loop, all inputs uploaded first
    md_g, pick_g, tgt_g, f_g = dev(md_rand), dev(pick), dev(tgt_rand), dev(f)
    cols = torch.arange(P + 1, device="cuda")
    t_g, o_g = dev(tokens), dev(offsets)
    st_g = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    long_g = torch.zeros(B, dtype=torch.int32, device="cuda")
    com_g = torch.full((B,), H + 1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    for s in range(steps):
        d_g, l_g, p_g, m_g = pkg.lookup_draft_ex(t_g, o_g, w.min_m, w.max_m, K)
        pkg.lookup_schedule(m_g, com_g, st_g, H, T, out=long_g)
        mdl = torch.where(pick_g[s][:, None], d_g[:, :H], md_g[s])
        blk_g, len_g, pm_g = pkg.lookup_fuse(d_g, m_g, mdl, long_g, H, T)
        prefix = cols[None, :] < f_g[s][:, None]
        target_g = tgt_g[s].clone()
        target_g[:, :P] = torch.where(prefix[:, :P], blk_g, target_g[:, :P])
        acc_g, commit_g, com_g = pkg.lookup_verify(blk_g, len_g, target_g)
        t_g, o_g = pkg.lookup_append(t_g, o_g, commit_g, com_g)
    d_g, l_g, p_g, m_g = pkg.lookup_draft_ex(t_g, o_g, w.min_m, w.max_m, K)
    np.testing.assert_array_equal(host(o_g), o_o)
    np.testing.assert_array_equal(host(t_g)[:o_o[-1]], t_o)
    np.testing.assert_array_equal(host(m_g), m_last)
    np.testing.assert_array_equal(host(d_g), d_last)


# ------------------------------------------------------- schedule, then fuse ----
@pytest.mark.parametrize("B,steps", [(1, 40), (33, 30), (4096, 12)])
@pytest.mark.parametrize("H,T,agree_n", [(7, 8, 2), (3, 2, 0), (16, 48, 3)])
@pytest.mark.parametrize("params", [dict(), dict(slack=0, enter_steps=1, sticky=0),
                                    dict(slack=3, enter_steps=3, sticky=5, tail_min=6)])
def test_plan_is_schedule_then_fuse(B, steps, H, T, agree_n, params):
    """lookup_plan over a scheduling trace against the oracle's schedule followed
    by its fuse with the new long flags: the long flags, the state, the block, its
    length and the point-mass flags, every step."""
    K = H + T + 2
    mlen, committed = gen.loop_schedule_trace(B, steps, H, T, seed=B + steps + H)
    st_o = np.zeros((B, 3), np.int32)
    st_g = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    tail_min = params.get("tail_min", 4)
    entered = 0
    for s in range(steps):
        ld, _, md, _ = gen.loop_fuse_inputs(B, K, H, T, agree_n, seed=100 * s + B)
        lg_o = oracle.schedule(mlen[s], committed[s], st_o, H, T, **params)
        want = oracle.fuse(ld, mlen[s], md, lg_o, H, T, agree_n=agree_n, tail_min=tail_min)
        lg_g, blk, ln, pm = pkg.lookup_plan(dev(ld), dev(mlen[s]), dev(md), dev(committed[s]), st_g, H, T,
                                            agree_n=agree_n, **params)
        np.testing.assert_array_equal(host(lg_g), lg_o, err_msg=f"long, step {s}")
        np.testing.assert_array_equal(host(st_g), st_o, err_msg=f"state, step {s}")
        for name, g, w in zip(("block", "len", "point mass"), (blk, ln, pm), want):
            np.testing.assert_array_equal(host(g), w, err_msg=f"{name}, step {s}")
        entered += int(lg_o.sum())
    if B > 1:
        assert 0 < entered < B * steps


@pytest.mark.parametrize("name", ["tiny", "chats"])
def test_decode_loop_with_plan_matches_oracle(name):
    """Draft -> plan (schedule + fuse) -> verify -> append, four steps, against the
    oracle's draft -> schedule -> fuse -> verify -> append."""
    w = gen.make_workload(name)
    B, H, T = w.B, 7, 8
    K = P = H + T
    tokens_o, offsets_o = w.tokens, w.offsets
    tokens_g, offsets_g = dev(w.tokens), dev(w.offsets)
    st_o = np.zeros((B, 3), np.int32)
    st_g = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    committed = np.full(B, H + 1, np.int32)
    com_g = dev(committed)
    for step in range(4):
        d_o, l_o, p_o, m_o = oracle.lookup_draft(tokens_o, offsets_o, w.min_m, w.max_m, K, threads=8)
        d_g, l_g, p_g, m_g = pkg.lookup_draft_ex(tokens_g, offsets_g, w.min_m, w.max_m, K)
        rng = gen.rng_for(step, 79)
        md = rng.integers(0, 50, size=(B, H), dtype=np.int64).astype(np.int32)
        pick = rng.random(B) < 0.33
        md[pick] = d_o[pick, :H]
        lg_o = oracle.schedule(m_o, committed, st_o, H, T)
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T)
        lg_g, blk_g, len_g, pm_g = pkg.lookup_plan(d_g, m_g, dev(md), com_g, st_g, H, T)
        for a, b in ((lg_o, lg_g), (blk_o, blk_g), (len_o, len_g), (pm_o, pm_g), (st_o, st_g)):
            np.testing.assert_array_equal(host(b), a)
        target = rng.integers(0, 50, size=(B, P + 1), dtype=np.int64).astype(np.int32)
        f = rng.integers(0, P + 1, size=B)
        for r in range(B):
            target[r, :f[r]] = blk_o[r, :f[r]]
        acc_o, com_o, nc_o = oracle.verify(blk_o, len_o, target)
        acc_g, com_t, nc_g = pkg.lookup_verify(blk_g, len_g, dev(target))
        np.testing.assert_array_equal(host(nc_g), nc_o)
        tokens_o, offsets_o = oracle.append(tokens_o, offsets_o, com_o, nc_o)
        tokens_g, offsets_g = pkg.lookup_append(tokens_g, offsets_g, com_t, nc_g)
        np.testing.assert_array_equal(host(offsets_g), offsets_o)
        np.testing.assert_array_equal(host(tokens_g)[:offsets_o[-1]], tokens_o)
        committed, com_g = nc_o, nc_g


# ------------------------------------------------- draft, then plan (two launches) ----
@pytest.mark.parametrize("name", ["tiny", "recitation25k", "periodic", "chats"])
def test_draft_plan_is_draft_then_plan(name):
    """lookup_draft_plan over a 4-step scheduling trace on a workload's histories,
    against the oracle's draft (K = H + T) -> schedule -> fuse: long flags, state,
    block, length, point masses, m and the draft length, every step."""
    w = gen.make_workload(name)
    B, H, T = w.B, 7, 8
    K = H + T
    t, o = dev(w.tokens), dev(w.offsets)
    d_o, l_o, p_o, m_o = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, K, threads=8)
    _, committed = gen.loop_schedule_trace(B, 4, H, T, seed=B + 5)
    st_o = np.zeros((B, 3), np.int32)
    st_g = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    for s in range(4):
        rng = gen.rng_for(s, 81)
        md = rng.integers(0, 50, size=(B, H), dtype=np.int64).astype(np.int32)
        pick = rng.random(B) < 0.4
        md[pick] = d_o[pick, :H]
        bump = pick & (rng.random(B) < 0.3)
        md[bump, 1] += 1                                 # agreement broken on the second token
        lg_o = oracle.schedule(m_o, committed[s], st_o, H, T)
        blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T)
        lg, blk, ln, pm, ml, dl = pkg.lookup_draft_plan(t, o, dev(md), dev(committed[s]), st_g, w.min_m, w.max_m,
                                                        H, T)
        for nm, g, e in (("long", lg, lg_o), ("state", st_g, st_o), ("block", blk, blk_o), ("len", ln, len_o),
                         ("point mass", pm, pm_o), ("mlen", ml, m_o), ("draft len", dl, l_o)):
            np.testing.assert_array_equal(host(g), e, err_msg=f"{nm}, step {s}")


@pytest.mark.parametrize("H,T,agree_n", [(3, 2, 3), (1, 0, 1), (16, 48, 2), (40, 24, 36)])
def test_draft_plan_block_shapes(H, T, agree_n):
    """Blocks of 5 to 64 positions (two tokens per lane past 32), agreement over
    up to 36 head tokens, min_m = 1 (dense matches) and histories of every short
    length with offsets[0] > 0."""
    rng = np.random.default_rng(H * 100 + T)
    lengths = rng.integers(0, 400, size=300)
    lengths[:20] = np.arange(20)
    lead = 3
    tokens = np.concatenate([rng.integers(0, 3, lead), rng.integers(0, 4, int(lengths.sum()))]).astype(np.int32)
    offsets = gen.offsets_from_lengths(lengths) + lead
    B, K = lengths.size, H + T
    d_o, l_o, p_o, m_o = oracle.lookup_draft(tokens, offsets, 1, 12, K, threads=8)
    md = rng.integers(0, 4, size=(B, H), dtype=np.int64).astype(np.int32)
    take = rng.random(B) < 0.5
    md[take] = np.where(d_o[take, :H] >= 0, d_o[take, :H], md[take])
    committed = rng.integers(1, H + T + 2, size=B).astype(np.int32)
    st_o = rng.integers(0, 2, size=(B, 3)).astype(np.int32)
    st_g = dev(st_o.copy())
    lg_o = oracle.schedule(m_o, committed, st_o, H, T)
    blk_o, len_o, pm_o = oracle.fuse(d_o, m_o, md, lg_o, H, T, agree_n=agree_n)
    lg, blk, ln, pm, ml, dl = pkg.lookup_draft_plan(dev(tokens), dev(offsets), dev(md), dev(committed), st_g, 1, 12,
                                                    H, T, agree_n=agree_n)
    for nm, g, e in (("long", lg, lg_o), ("state", st_g, st_o), ("block", blk, blk_o), ("len", ln, len_o),
                     ("point mass", pm, pm_o), ("mlen", ml, m_o), ("draft len", dl, l_o)):
        np.testing.assert_array_equal(host(g), e, err_msg=nm)


# ------------------------------------------------------ draft-source controller ----
@pytest.mark.parametrize("B", [1, 7, 4096])
@pytest.mark.parametrize("params", [
    dict(n_lookup=7, n_model=3, t_lookup=1.3, t_model=1.1, t_plain=0.77, alpha=0.125, margin=0.05),
    dict(n_lookup=15, n_model=3, t_lookup=2.9, t_model=1.0, t_plain=0.9, alpha=0.3, margin=0.0, edges=(5, 7, 9)),
    dict(n_lookup=4, n_model=0, t_lookup=1.0, t_model=0.5, t_plain=0.4, alpha=1.0, margin=0.25, edges=(4, 4, 12)),
])
def test_policy_matches_oracle_bit_for_bit(B, params):
    """lookup_policy over a 40-step trace with random match lengths, accepted counts
    (some outside [0, drafted]) and priors: the choices, the integer state and
    every float of the acceptance estimates equal the oracle's exactly."""
    steps = 40
    rng = gen.rng_for(B * 31 + len(params), 90)
    acc_o = rng.uniform(0.0, 1.0, size=(B, 5)).astype(np.float32)
    prev_o = np.zeros((B, 3), np.int32)
    acc_g, prev_g = dev(acc_o.copy()), dev(prev_o.copy())
    seen = set()
    for s in range(steps):
        m = np.where(rng.random(B) < 0.3, 0, rng.integers(3, 15, size=B)).astype(np.int32)
        accepted = rng.integers(-1, 18, size=B).astype(np.int32)
        want = oracle.policy(m, accepted, acc_o, prev_o, **params)
        got = pkg.lookup_policy(dev(m), dev(accepted), acc_g, prev_g, **params)
        np.testing.assert_array_equal(host(got), want, err_msg=f"choice, step {s}")
        np.testing.assert_array_equal(host(prev_g), prev_o, err_msg=f"prev, step {s}")
        a = host(acc_g)
        assert np.array_equal(a.view(np.uint32), acc_o.view(np.uint32)), f"acceptance bits, step {s}"
        seen.update(int(c) for c in want)
    if B > 1:
        assert len(seen) >= 2                        # the trace switches between choices
