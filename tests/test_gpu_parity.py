"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Every comparison is bit-exact on out_len, out_pos, the match length and all K
draft slots (the sentinels included), on the same seeded inputs.  Covered:
the five synthetic workloads at full size (default seeds and five more each),
the hand-worked fixtures, and edge cases: empty batch, short and empty
requests, K = 0 and the largest K, the widest m range, unaligned token
pointers, offsets[0] > 0, fewer tokens than scan CTAs, more requests than the
offsets the scan keeps in shared memory, all-equal and tiny-alphabet histories,
long single requests spread over many CTAs, a match ending exactly at a tile or
chunk boundary, clusters of dozens of requests starting inside one quad, batch
sizes on both sides of the switch to the lane-per-request fill (with requests
spanning hundreds of scan warps), the staged and host-buffer entry points
(page-locked inputs at every 4-byte phase, mixed and pageable inputs), the
read-floor measurement aid, repeated calls and the failure path of the bounded
waits.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle
from goldens import load_cases

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytestmark = [pytest.mark.gpu, pytest.mark.skip(reason="needs a CUDA GPU")]

import prompt_lookup_speculative_gb300 as pkg  # noqa: E402

DEV = "cuda:0"


def run_gpu(tokens: np.ndarray, offsets: np.ndarray, min_m, max_m, K, token_pad: int = 0):
    """Run lookup_draft_ex; token_pad shifts the tokens pointer by that many int32."""
    buf = torch.zeros(tokens.size + token_pad + 4, dtype=torch.int32, device=DEV)
    buf[token_pad:token_pad + tokens.size] = torch.from_numpy(tokens).to(DEV)
    t = buf[token_pad:token_pad + tokens.size] if tokens.size else buf[token_pad:token_pad]
    o = torch.from_numpy(np.ascontiguousarray(offsets, np.int64)).to(DEV)
    d, ln, p, m = pkg.lookup_draft_ex(t, o, min_m, max_m, K)
    torch.cuda.synchronize()
    return d.cpu().numpy(), ln.cpu().numpy(), p.cpu().numpy(), m.cpu().numpy()


def assert_parity(tokens, offsets, min_m, max_m, K, token_pad=0, threads=8):
    got = run_gpu(tokens, offsets, min_m, max_m, K, token_pad)
    want = oracle.lookup_draft(tokens, offsets, min_m, max_m, K, threads=threads)
    for name, g, w in zip(("draft", "len", "pos", "mlen"), got, want):
        if not np.array_equal(g, w):
            bad = np.nonzero((g != w).reshape(g.shape[0], -1).any(axis=1))[0] if g.ndim else []
            raise AssertionError(f"{name} differs at requests {list(bad[:10])} "
                                 f"(gpu {g[bad[:3]]}, oracle {w[bad[:3]]})")
    return got


@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_workload_default_seed(name):
    w = gen.make_workload(name)
    assert_parity(w.tokens, w.offsets, w.min_m, w.max_m, w.K)


@pytest.mark.parametrize("seed", [6, 7, 8, 9, 10])
@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_workload_more_seeds(name, seed):
    w = gen.make_workload(name, seed)
    assert_parity(w.tokens, w.offsets, w.min_m, w.max_m, w.K)


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c.name)
def test_hand_worked(case):
    d, ln, p, m = run_gpu(case.tokens, case.offsets, case.min_m, case.max_m, case.K)
    np.testing.assert_array_equal(m, case.expect_m)
    np.testing.assert_array_equal(p, case.expect_pos)
    np.testing.assert_array_equal(ln, case.expect_len)
    np.testing.assert_array_equal(d, case.expect_draft)


def test_empty_batch():
    t = torch.zeros(0, dtype=torch.int32, device=DEV)
    o = torch.zeros(1, dtype=torch.int64, device=DEV)
    d, ln, p = pkg.lookup_draft(t, o, 4, 12, 15)
    assert d.shape == (0, 15) and ln.numel() == 0


@pytest.mark.parametrize("pad", [0, 1, 2, 3])
def test_unaligned_tokens_pointer(pad):
    w = gen.make_workload("periodic", 11)
    assert_parity(w.tokens, w.offsets, w.min_m, w.max_m, w.K, token_pad=pad)


@pytest.mark.parametrize("pad", [0, 1, 3])
def test_short_requests_and_offset_base(pad):
    """Lengths 0, 1, min_m, min_m + 1 and a few longer ones, all tokens equal, with
    offsets[0] > 0 (tokens before it belong to no request)."""
    rng = np.random.default_rng(pad)
    lengths = [0, 1, 4, 5, 0, 13, 12, 3, 100, 0, 6, 1]
    lead = 7
    tokens = np.concatenate([rng.integers(0, 3, lead), np.full(sum(lengths), 5)]).astype(np.int32)
    offsets = gen.offsets_from_lengths(lengths) + lead
    assert_parity(tokens, offsets, 4, 12, 15, token_pad=pad)


@pytest.mark.parametrize("K", [0, 1, 31, 32, 33, 64])
def test_draft_lengths(K):
    w = gen.make_workload("periodic", 12)
    assert_parity(w.tokens, w.offsets, w.min_m, w.max_m, K)


@pytest.mark.parametrize("min_m,max_m", [(1, 1), (1, 32), (32, 32), (4, 4), (2, 9), (12, 12)])
def test_m_ranges(min_m, max_m):
    rng = np.random.default_rng(min_m * 100 + max_m)
    lengths = rng.integers(0, 3000, size=40)
    tokens = rng.integers(0, 4, size=int(lengths.sum())).astype(np.int32)
    assert_parity(tokens, gen.offsets_from_lengths(lengths), min_m, max_m, 9)


def test_fewer_tokens_than_ctas():
    """A handful of tokens: most scan CTAs get an empty chunk."""
    tokens = np.array([1, 2, 3, 1, 2, 3, 1, 2, 9, 9, 9, 9, 9, 4, 4, 4, 4, 4, 4], dtype=np.int32)
    offsets = np.array([0, 8, 8, 13, 19], dtype=np.int64)
    for pad in range(4):
        assert_parity(tokens, offsets, 2, 4, 5, token_pad=pad)
        assert_parity(tokens, offsets, 1, 3, 3, token_pad=pad)


@pytest.mark.parametrize("B", [4096, 4097, 10000])
def test_many_requests(B):
    """Around and above the number of offsets the scan keeps in shared memory."""
    rng = np.random.default_rng(B)
    lengths = rng.integers(0, 40, size=B)
    tokens = rng.integers(0, 3, size=int(lengths.sum())).astype(np.int32)
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 2, 6, 5)


def test_many_requests_long_chunks():
    rng = np.random.default_rng(5)
    lengths = rng.integers(0, 600, size=6000)
    tokens = rng.integers(0, 50, size=int(lengths.sum())).astype(np.int32)
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 2, 12, 7)


def clustered_lengths(rng, B, cluster):
    """Long requests separated by runs of `cluster` empty or 1-3 token requests, so
    that dozens of requests start inside one 4-token quad."""
    lengths = []
    while len(lengths) < B:
        lengths.append(int(rng.integers(200, 6000)))
        lengths.extend(int(x) for x in rng.choice([0, 0, 0, 1, 2, 3], size=cluster))
    return np.array(lengths[:B])


@pytest.mark.parametrize("cluster", [1, 5, 40, 70])
@pytest.mark.parametrize("pad", [0, 1, 2, 3])
def test_clustered_short_requests(cluster, pad):
    """Long requests separated by up to 70 requests that start inside one quad, in
    batches for either fill."""
    rng = np.random.default_rng(cluster * 10 + pad)
    lengths = clustered_lengths(rng, 400 if pad % 2 == 0 else 1500, cluster)
    tokens = rng.integers(0, 3, size=int(lengths.sum())).astype(np.int32)
    offsets = gen.offsets_from_lengths(lengths) + int(rng.integers(0, 4))
    tokens = np.concatenate([np.full(int(offsets[0]), 1, np.int32), tokens])
    assert_parity(tokens, offsets, 1, 12, 5, token_pad=pad)
    assert_parity(tokens, offsets, 4, 12, 7, token_pad=pad)


@pytest.mark.parametrize("B", [2, 9, 300, 1023, 1024, 1025, 2432])
def test_log_uniform_lengths(B):
    """Log-uniform lengths (a few long requests, many boundaries), on both sides of
    the batch size from which the fill takes one request per lane."""
    rng = np.random.default_rng(B)
    lengths = np.exp(rng.uniform(0, np.log(40000), size=B)).astype(np.int64)
    tokens = rng.integers(0, 6, size=int(lengths.sum())).astype(np.int32)
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 4, 12, 9, token_pad=B % 4)


@pytest.mark.parametrize("B", [1023, 1024, 3000])
def test_large_batch_with_long_requests(B):
    """Around the batch size from which the fill takes one request per lane, with
    a few requests long enough to span hundreds of scan warps (those are folded
    by the whole warp)."""
    rng = np.random.default_rng(B + 77)
    lengths = rng.integers(0, 300, size=B)
    lengths[rng.choice(B, size=5, replace=False)] = rng.integers(100_000, 600_000, size=5)
    tokens = rng.integers(0, 3, size=int(lengths.sum())).astype(np.int32)
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 4, 12, 9, token_pad=B % 4)


@pytest.mark.parametrize("S", [511, 512, 2047, 2048])
def test_chunk_size_at_range_count_switch(S):
    """Batches whose scan CTA chunk is exactly S quads on this GPU's SM count: 511 /
    512 quads (8 or 12 warp ranges per CTA) and 2047 / 2048 (12 or 16), where the
    scan's multiply-high split and the fill's division must agree."""
    G = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(S)
    for nq in ((S - 1) * G + 1, S * G):
        cuts = np.sort(rng.integers(0, 4 * nq - 1, size=int(rng.integers(20, 90))))
        offsets = np.concatenate([[0], cuts, [4 * nq - 1]]).astype(np.int64)
        tokens = rng.integers(0, 40, size=4 * nq - 1).astype(np.int32)
        for r in range(0, offsets.size - 1, 3):              # planted copies of earlier spans
            o, n = int(offsets[r]), int(offsets[r + 1])
            if n - o > 64:
                c = int(rng.integers(13, min(60, (n - o) // 2)))
                s0 = int(rng.integers(o, n - 2 * c))
                tokens[n - c:n] = tokens[s0:s0 + c]
        assert_parity(tokens, offsets, 4, 12, 15)


def test_all_equal_tokens():
    lengths = [1, 17, 4096, 25000, 3]
    tokens = np.full(sum(lengths), -7, dtype=np.int32)
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 4, 12, 15)


@pytest.mark.parametrize("alphabet", [2, 3, 5])
def test_tiny_alphabet_dense_matches(alphabet):
    rng = np.random.default_rng(alphabet)
    lengths = rng.integers(0, 20000, size=50)
    tokens = rng.integers(0, alphabet, size=int(lengths.sum())).astype(np.int32)
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 4, 12, 15)


def test_extreme_token_values():
    rng = np.random.default_rng(3)
    vals = np.array([np.iinfo(np.int32).min, np.iinfo(np.int32).max, -1, 0], dtype=np.int32)
    lengths = rng.integers(1, 5000, size=30)
    tokens = vals[rng.integers(0, 4, size=int(lengths.sum()))]
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 3, 10, 6)


def test_long_single_request():
    """One 3M-token history shared by every scan CTA; matches planted near its start."""
    rng = np.random.default_rng(11)
    L = 3_000_000
    t = rng.integers(0, 1 << 30, size=L).astype(np.int32)
    t[-20:] = t[100:120]          # the only 12-gram repeat: p = 108
    got = assert_parity(t, np.array([0, L], np.int64), 4, 12, 15)
    assert got[2][0] == 108 and got[3][0] == 12


@pytest.mark.parametrize("where", range(0, 64, 5))
def test_match_end_at_every_alignment(where):
    """Move a planted match across quad, tile and chunk boundaries."""
    rng = np.random.default_rng(where)
    L = 200_000
    t = rng.integers(0, 1 << 30, size=L).astype(np.int32)
    src = 16384 * 3 + where - 12     # ends near a multiple of the 16 KB tile
    t[-12:] = t[src:src + 12]
    lengths = [L, 5000, 1 + where]
    tokens = np.concatenate([t, rng.integers(0, 7, size=5001 + where).astype(np.int32)])
    assert_parity(tokens, gen.offsets_from_lengths(lengths), 4, 12, 15, token_pad=where % 4)


def test_cross_request_boundary():
    rng = np.random.default_rng(7)
    a = rng.integers(0, 1 << 20, size=3000).astype(np.int32)
    b = rng.integers(0, 1 << 20, size=3000).astype(np.int32)
    b[-12:] = a[-12:]
    tokens = np.concatenate([a, b])
    offsets = np.array([0, a.size, a.size + b.size], dtype=np.int64)
    d, ln, p, m = assert_parity(tokens, offsets, 4, 12, 5)
    assert ln[1] == 0


def test_staged_entry_points_match_one_call():
    w = gen.make_workload("recitation25k")
    t = torch.from_numpy(w.tokens).to(DEV)
    o = torch.from_numpy(w.offsets).to(DEV)
    ws = torch.empty(pkg.workspace_bytes(w.B), dtype=torch.uint8, device=DEV)
    ws.fill_(0xAB)                      # garbage: the scan must not need a clean workspace
    pkg.lookup_draft_scan(t, o, w.min_m, w.max_m, ws)
    d1, l1, p1, m1 = pkg.lookup_draft_fill(t, o, w.min_m, w.max_m, w.K, ws, with_mlen=True)
    d2, l2, p2, m2 = pkg.lookup_draft_ex(t, o, w.min_m, w.max_m, w.K)
    torch.cuda.synchronize()
    for a, b in ((d1, d2), (l1, l2), (p1, p2), (m1, m2)):
        assert torch.equal(a, b)


def test_host_entry_point():
    w = gen.make_workload("chats", 13)
    d, ln, p = pkg.lookup_draft_host(w.tokens, w.offsets, w.min_m, w.max_m, w.K)
    od, oln, op, _ = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8)
    np.testing.assert_array_equal(d, od)
    np.testing.assert_array_equal(ln, oln)
    np.testing.assert_array_equal(p, op)


@pytest.mark.parametrize("pinned", ["all", "some", "none"])
def test_host_entry_point_pinned_outputs(pinned):
    """Page-locked outputs are written by the fill kernel directly; mixed or
    pageable outputs go through copies.  Same results either way."""
    w = gen.make_workload("recitation25k", 15)
    B, K = w.B, w.K
    def buf(shape, pin):
        t = torch.full(shape, -77, dtype=torch.int32)
        return t.pin_memory() if pin else t
    out = (buf((B, K), pinned != "none"), buf((B,), pinned == "all"), buf((B,), pinned != "none"))
    tok = torch.from_numpy(w.tokens).pin_memory()
    off = torch.from_numpy(w.offsets).pin_memory()
    d, ln, p = pkg.lookup_draft_host(tok, off, w.min_m, w.max_m, K, out=out)
    od, oln, op, _ = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, K, threads=8)
    np.testing.assert_array_equal(d.numpy(), od)
    np.testing.assert_array_equal(ln.numpy(), oln)
    np.testing.assert_array_equal(p.numpy(), op)


def test_host_entry_point_offset_base():
    tokens = np.array([9, 9, 9, 1, 2, 3, 1, 2, 3, 1, 2], dtype=np.int32)
    offsets = np.array([3, 3, 11], dtype=np.int64)
    d, ln, p = pkg.lookup_draft_host(tokens, offsets, 2, 4, 4)
    od, oln, op, _ = oracle.lookup_draft(tokens, offsets, 2, 4, 4)
    np.testing.assert_array_equal(d, od)
    np.testing.assert_array_equal(ln, oln)
    np.testing.assert_array_equal(p, op)


@pytest.mark.parametrize("first", [0, 5])
@pytest.mark.parametrize("shift", [0, 1, 2, 3])
def test_host_entry_point_pinned_inputs_any_phase(shift, first):
    """Page-locked inputs are read by the device straight from host memory, in
    whole 16-byte units of their address range: tokens starting at any 4-byte
    phase, and offsets[0] > 0, give the oracle's results."""
    w = gen.make_workload("periodic", 16 + shift)
    n = w.tokens.shape[0]
    big = torch.full((shift + first + n + 8,), 7, dtype=torch.int32).pin_memory()
    tok = big[shift: shift + first + n]
    tok[first:] = torch.from_numpy(w.tokens)
    off = torch.from_numpy(w.offsets + first).pin_memory()
    d, ln, p = pkg.lookup_draft_host(tok, off, w.min_m, w.max_m, w.K)
    od, oln, op, _ = oracle.lookup_draft(tok.numpy(), off.numpy(), w.min_m, w.max_m, w.K, threads=8)
    np.testing.assert_array_equal(d, od)
    np.testing.assert_array_equal(ln, oln)
    np.testing.assert_array_equal(p, op)


@pytest.mark.parametrize("pin", ["tokens", "offsets"])
def test_host_entry_point_mixed_inputs(pin):
    """One input page-locked and the other pageable: both go through copies."""
    w = gen.make_workload("ragged262k", 17)
    tok = torch.from_numpy(w.tokens)
    off = torch.from_numpy(w.offsets)
    tok = tok.pin_memory() if pin == "tokens" else tok
    off = off.pin_memory() if pin == "offsets" else off
    d, ln, p = pkg.lookup_draft_host(tok, off, w.min_m, w.max_m, w.K)
    od, oln, op, _ = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8)
    np.testing.assert_array_equal(d, od)
    np.testing.assert_array_equal(ln, oln)
    np.testing.assert_array_equal(p, op)


def test_host_entry_point_pinned_empty_histories():
    tok = torch.arange(5, dtype=torch.int32).pin_memory()
    off = torch.tensor([3, 3, 3], dtype=torch.int64).pin_memory()
    d, ln, p = pkg.lookup_draft_host(tok, off, 4, 12, 3)
    np.testing.assert_array_equal(ln, [0, 0])
    np.testing.assert_array_equal(p, [-1, -1])
    np.testing.assert_array_equal(d, np.full((2, 3), -1, np.int32))


@pytest.mark.parametrize("shape", [(1, 32), (2, 512), (4, 256), (8, 256), (0, 0)])
def test_read_floor_streams_without_writing(shape):
    """The measurement aid reads its bytes and leaves the output word alone unless
    their fold hits its fixed pattern (the XOR of 0 .. 2^20 - 1 is 0)."""
    x = torch.arange(1 << 20, dtype=torch.int32, device=DEV)
    out = torch.full((1,), 123, dtype=torch.int32, device=DEV)
    pkg.read_floor(x, *shape, out=out)
    pkg.read_floor(x[:4], *shape, out=out)                   # fewer 16-byte units than threads
    torch.cuda.synchronize()
    assert out.item() == 123


@pytest.mark.parametrize("n16", [3, 193, (3 << 16) + 3, (41 << 16) + 1])
def test_bulk_read_floor_odd_sizes(n16):
    """The bulk read over sizes whose warp ranges and tiles end unevenly (48 bytes,
    one tile and a quad, 3 MB + 48 bytes, 41 MB + 16 bytes): it completes and
    leaves the output word alone."""
    x = torch.zeros(4 * n16, dtype=torch.int32, device=DEV)
    x[::7] = 1
    out = torch.full((1,), 123, dtype=torch.int32, device=DEV)
    pkg.read_floor(x, 0, 0, out=out)
    torch.cuda.synchronize()
    assert out.item() == 123


def test_bulk_read_floor_wait_runs_out_cleanly():
    """With a 1 ns wait limit the bulk read's warps give up at their first tile,
    store -1, let their copies land (bounded by 1 s, not by the limit) and stop;
    the context stays usable and the next read with the default limit is clean."""
    x = torch.arange(1 << 24, dtype=torch.int32, device=DEV)      # 64 MB
    out = torch.full((1,), 123, dtype=torch.int32, device=DEV)
    try:
        pkg.set_wait_limit_ns(1)
        pkg.read_floor(x, 0, 0, out=out)
        torch.cuda.synchronize()
    finally:
        pkg.set_wait_limit_ns(0)
    assert out.item() == -1
    out.fill_(123)
    pkg.read_floor(x, 0, 0, out=out)
    torch.cuda.synchronize()
    assert out.item() == 123
    w = gen.make_workload("tiny", 19)
    assert_parity(w.tokens, w.offsets, w.min_m, w.max_m, w.K)


def test_repeated_calls_and_streams():
    w = gen.make_workload("ragged262k", 14)
    t = torch.from_numpy(w.tokens).to(DEV)
    o = torch.from_numpy(w.offsets).to(DEV)
    ref = pkg.lookup_draft(t, o, w.min_m, w.max_m, w.K)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(5):
            outs.append(pkg.lookup_draft(t, o, w.min_m, w.max_m, w.K))
    torch.cuda.synchronize()
    for out in outs:
        for a, b in zip(out, ref):
            assert torch.equal(a, b)
    want = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8)
    np.testing.assert_array_equal(ref[0].cpu().numpy(), want[0])


def test_bounded_waits_fail_cleanly():
    """With a 1 ns wait limit the scan's bounded waits run out.  A CTA whose wait
    for its TMA copy of the offsets runs out reads them from global memory
    instead; one whose wait for a history tile runs out lets its copies land,
    marks its requests LOOKUP_DRAFT_LEN_FAILED and returns.  Every request is
    then either exactly the oracle's or marked failed, and the next call with
    the default limit is exact again (the context stays usable)."""
    w = gen.make_workload("ragged262k", 15)
    t = torch.from_numpy(w.tokens).to(DEV)
    o = torch.from_numpy(w.offsets).to(DEV)
    want = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8)
    try:
        pkg.set_wait_limit_ns(1)
        d, ln, p, m = pkg.lookup_draft_ex(t, o, w.min_m, w.max_m, w.K)
        torch.cuda.synchronize()
    finally:
        pkg.set_wait_limit_ns(0)
    d, ln, p, m = (x.cpu().numpy() for x in (d, ln, p, m))
    ok = ln != pkg.LEN_FAILED
    np.testing.assert_array_equal(ln[ok], want[1][ok])
    np.testing.assert_array_equal(p[ok], want[2][ok])
    np.testing.assert_array_equal(d[ok], want[0][ok])
    assert np.all(p[~ok] == -1) and np.all(d[~ok] == -1)
    got = run_gpu(w.tokens, w.offsets, w.min_m, w.max_m, w.K)
    for g, exp in zip(got, want):
        np.testing.assert_array_equal(g, exp)


def test_cuda_error_inside_capture_is_reported_and_the_context_stays_usable():
    """lookup_draft_host called inside a stream capture: its copy from pageable host
    memory and its stream synchronisation are not allowed there, so the call
    returns LOOKUP_DRAFT_ECUDA with the failing call named, and the capture ends
    in an error.  Nothing was executed on the device; the next call is exact."""
    lib = pkg.load_library()
    w = gen.make_workload("tiny", 18)
    assert_parity(w.tokens, w.offsets, w.min_m, w.max_m, w.K)       # device set up outside the capture
    out_d = np.zeros(w.B * w.K, np.int32)
    out_l, out_p = np.zeros(w.B, np.int32), np.zeros(w.B, np.int32)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    seen = []
    with pytest.raises(Exception):
        with torch.cuda.graph(g, stream=s):
            rc = lib.lookup_draft_host(w.tokens.ctypes.data, w.offsets.ctypes.data, w.B, w.min_m, w.max_m, w.K,
                                       out_d.ctypes.data, out_l.ctypes.data, out_p.ctypes.data,
                                       torch.cuda.current_stream().cuda_stream)
            seen.append((rc, lib.lookup_draft_last_cuda_error().decode()))
    assert seen and seen[0][0] == -2, seen
    assert "cuda" in seen[0][1], seen
    del g
    torch.cuda.synchronize()
    assert_parity(w.tokens, w.offsets, w.min_m, w.max_m, w.K)
