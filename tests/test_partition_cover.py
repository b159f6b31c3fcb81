"""CPU emulation of the scan's work split: partition, tiles, halos, slots, cover.

The scan kernel (csrc/lookup_draft.cu) cuts the batch into CTA chunks and warp
ranges with 32-bit arithmetic (the division by the grid size done as a
multiply-high by a host-computed reciprocal), copies each range in tiles with a
halo of earlier quads, keeps each (warp, request) result in slot v + r, and the
fill finds a request's slots from the partition alone.  This test restates that
integer arithmetic in Python, with the kernel's constants read from its source,
and checks on random batches that

- the division by the grid size is exact for every value the kernel divides;
- a chunk is never shorter than kChunkMin quads, so a small batch leaves the
  last CTAs empty;
- the warp ranges tile the batch's quads, so every candidate end of every
  request (positions min_m - 1 .. L - 2) is examined by exactly one warp;
- every tile's halo reaches max_m - 1 tokens before the tile (or the batch
  start), and every copy fits its shared-memory buffer;
- slot indices never collide, and the fill's cover of a request is exactly the
  set of warps whose range meets it.
No GPU is needed; the GPU parity tests check the kernel itself.
"""
from __future__ import annotations

import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "prompt_lookup_speculative_gb300", "csrc", "lookup_draft.cu")).read()
HDR = open(os.path.join(ROOT, "include", "lookup_draft.h")).read()


def _const(name, text=SRC):
    m = re.search(r"constexpr int " + name + r"\s*=\s*(\d+);", text)
    assert m, name
    return int(m.group(1))


K_WARPS = _const("kWarps")
CHUNK_MIN = _const("kChunkMin")
CHUNK_SMALL = _const("kChunkSmall")
CHUNK_MID = _const("kChunkMid")
K_BUFS = _const("kBufs")
TQ_MAX = _const("kTileQuadsMax")
TQ_MIN = _const("kTileQuadsMin")
HALO_QUADS = _const("kHaloQuads")
MAX_M = int(re.search(r"#define LOOKUP_DRAFT_MAX_M\s+(\d+)", HDR).group(1))
BUF_QUADS = TQ_MAX + HALO_QUADS


def grid_divider(G):
    """The host's reciprocal for floor(n / G), n < 2^31."""
    if G <= 1:
        return 0, -1
    l = 0
    while (1 << l) < G:
        l += 1
    k = 31 + l
    return ((1 << k) + G - 1) // G, k - 32


def div_grid(n, magic, shift):
    return n if shift < 0 else ((n * magic) >> 32) >> shift


@pytest.mark.parametrize("G", [1, 2, 3, 7, 76, 128, 132, 148, 152, 160, 264, 1024])
def test_grid_division_is_exact(G):
    magic, shift = grid_divider(G)
    assert shift < 0 or magic < (1 << 32)
    rng = np.random.default_rng(G)
    ns = [0, 1, G - 1, G, G + 1, (1 << 31) - 1, (1 << 31) - G]
    ns += [int(x) for x in rng.integers(0, 1 << 31, size=4000)]
    ns += [q * G + r for q in ((1 << 31) // G - 1, (1 << 31) // G - 2) for r in (0, G - 1) if q * G + r < (1 << 31)]
    for n in ns:
        assert div_grid(n, magic, shift) == n // G, (G, n)


def warp_span(S):
    """Quads per warp range of a chunk of S quads: 8 ranges below CHUNK_SMALL,
    12 below CHUNK_MID, else K_WARPS (the kernel's warp_span32)."""
    w = 8 if S < CHUNK_SMALL else (12 if S < CHUNK_MID else K_WARPS)
    return (S + w - 1) // w


def warp_ranges(nq, G):
    """[lo, hi) per virtual chunk v = c * K_WARPS + w, quads relative to q_lo."""
    magic, shift = grid_divider(G)
    S = max(div_grid(nq + G - 1, magic, shift), CHUNK_MIN)
    Sw = warp_span(S)
    out = []
    for c in range(G):
        c0 = c * S
        c1 = min(c0 + S, nq)
        for w in range(K_WARPS):
            lo = c0 + w * Sw
            out.append((lo, min(lo + Sw, c1)))
    return S, Sw, out


def fill_partition(nq, G):
    """(S, Sw) as the fill kernel forms them (make_partition: plain divisions, the
    wide-chunk rule written separately), to be held against the scan's."""
    S = max((nq + G - 1) // G, CHUNK_MIN)
    Sw = warp_span(S) if S < CHUNK_MID else (S + K_WARPS - 1) // K_WARPS
    return S, Sw


def tiles(wn):
    tq = wn if wn <= TQ_MAX else (wn + 1) // 2
    tq = min(max(tq, TQ_MIN), TQ_MAX)
    ntiles = (wn + TQ_MAX - 1) // TQ_MAX if tq == TQ_MAX else (2 if wn > tq else 1)
    assert ntiles == -(-wn // tq)                       # the kernel's division-free count
    return tq, ntiles


def owner(offa, e):
    """The request holding element e (largest r with offa[r] <= e)."""
    return int(np.searchsorted(offa[:-1], e, side="right")) - 1


def emulate(offsets, shift, G, min_m, max_m):
    B = len(offsets) - 1
    offa = np.asarray(offsets, np.int64) + shift
    a_begin, a_end = int(offa[0]), int(offa[B])
    if a_end <= a_begin:
        return
    q_lo = a_begin >> 2
    nq = ((a_end + 3) >> 2) - q_lo
    S, Sw, ranges = warp_ranges(nq, G)
    assert (S, Sw) == fill_partition(nq, G)              # scan and fill agree on the split
    halo = (max_m - 1 + 3) >> 2
    assert halo <= HALO_QUADS
    covered = np.zeros(nq, np.int32)
    slots = {}
    touching = {}
    for v, (lo, hi) in enumerate(ranges):
        if lo >= hi:
            continue
        covered[lo:hi] += 1
        wn = hi - lo
        tq, ntiles = tiles(wn)
        lead = min(halo, lo)
        for k in range(ntiles):
            t0 = k * tq
            t1 = min(t0 + tq, wn)
            ls = max(t0 - halo, -lead)
            assert t1 - ls <= BUF_QUADS                  # the copy fits its buffer
            assert HALO_QUADS - (t0 - ls) >= 0
            first = 4 * (q_lo + lo + t0)                 # the tile's first element
            ctx = 4 * (q_lo + lo + ls)                   # the copy's first element
            assert ctx <= max(first - (max_m - 1), 4 * q_lo)
            assert q_lo + lo + ls >= q_lo
        WA = 4 * (q_lo + lo)
        wbeg = max(WA, a_begin) - WA
        wend = min(4 * (q_lo + hi), a_end) - WA
        rw_lo, rw_hi = owner(offa, WA + wbeg), owner(offa, WA + wend - 1)
        for r in range(rw_lo, rw_hi + 1):
            if offa[r + 1] > offa[r]:
                assert v + r not in slots, "slot collision"
                assert v + r < B + G * K_WARPS
                slots[v + r] = (v, r)
                touching.setdefault(r, []).append(v)
    assert (covered == 1).all()                          # the ranges tile the batch
    for r in range(B):
        o, n = int(offa[r]), int(offa[r + 1])
        if n <= o:
            continue
        # every candidate end lies in some warp's range (covered once, above)
        for q in (o + min_m - 1, n - 2):
            if o + min_m - 1 <= q <= n - 2:
                assert 0 <= (q >> 2) - q_lo < nq
        # the fill's cover: the warps holding the request's first and last quads
        def vchunk_of_quad(x):
            c = x // S
            return c * K_WARPS + (x - c * S) // Sw
        v0 = vchunk_of_quad((o >> 2) - q_lo)
        v1 = vchunk_of_quad(((n - 1) >> 2) - q_lo)
        want = touching.get(r, [])
        got = [v for v in range(v0, v1 + 1) if ranges[v][0] < ranges[v][1]]
        assert got == want, (r, got[:4], want[:4])


def random_offsets(rng):
    B = int(rng.choice([1, 2, 5, 17, 64, 200]))
    kind = rng.random()
    if kind < 0.3:
        lengths = rng.choice([0, 0, 1, 2, 3, 4, 5, 9, 13], size=B)
    elif kind < 0.6:
        lengths = np.exp(rng.uniform(0, np.log(60000), size=B)).astype(np.int64)
    else:
        lengths = rng.integers(0, 5000, size=B)
    lead = int(rng.integers(0, 9))
    return np.concatenate([[lead], lead + np.cumsum(lengths)]).astype(np.int64)


@pytest.mark.parametrize("G", [152, 7, 2, 1])
@pytest.mark.parametrize("seed", range(5))
def test_work_split_covers_every_candidate_once(G, seed):
    rng = np.random.default_rng(1000 * G + seed)
    for _ in range(8):
        emulate(random_offsets(rng), int(rng.integers(0, 4)), G, 4, 12)
        emulate(random_offsets(rng), int(rng.integers(0, 4)), G, 1, MAX_M)


def test_workload_sized_batches():
    # the five workloads' shapes on 152 SMs: one long, many short, ragged
    for lengths in ([25_000] * 64, [2048] * 4096, [4096] * 8, [8192] * 64,
                    np.exp(np.random.default_rng(4).uniform(np.log(512), np.log(262_144), size=256)).astype(np.int64)):
        offsets = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
        emulate(offsets, 0, 152, 4, 12)


def batch_with_chunk(S, G, rng, shift=0, lead=0):
    """Offsets of a batch whose CTA chunk is exactly S quads on G CTAs: its quads
    run from (S - 1) * G + 1 to S * G (both ends are drawn), cut into requests of
    random lengths (some empty, some shorter than a quad)."""
    nq = int(rng.choice([(S - 1) * G + 1, S * G, int(rng.integers((S - 1) * G + 1, S * G + 1))]))
    a0 = 4 * ((lead + shift) >> 2)
    total = 4 * nq - ((lead + shift) - a0) - int(rng.integers(0, 4))
    cuts = np.sort(rng.integers(0, total + 1, size=int(rng.integers(0, 60))))
    bounds = np.concatenate([[0], cuts, [total]])
    return (lead + bounds).astype(np.int64)


@pytest.mark.parametrize("S", [CHUNK_SMALL - 1, CHUNK_SMALL, CHUNK_MID - 1, CHUNK_MID])
@pytest.mark.parametrize("G", [152, 148, 7])
def test_chunk_sizes_at_the_range_count_switches(S, G):
    """A CTA chunk of 511 / 512 quads (8 or 12 warp ranges) and of 2047 / 2048 (12 or
    16): the scan's multiply-high path and the fill's division give the same split,
    and the ranges still tile the batch with an exact cover per request."""
    rng = np.random.default_rng(S * 1000 + G)
    for _ in range(6):
        shift = int(rng.integers(0, 4))
        lead = int(rng.integers(0, 9))
        offsets = batch_with_chunk(S, G, rng, shift, lead)
        offa = offsets + shift
        q_lo = int(offa[0]) >> 2
        nq = ((int(offa[-1]) + 3) >> 2) - q_lo
        assert warp_ranges(nq, G)[0] == S
        emulate(offsets, shift, G, 4, 12)
        emulate(offsets, shift, G, 1, MAX_M)


@pytest.mark.parametrize("G", [152, 7])
def test_small_batches_use_whole_minimum_chunks(G):
    """Batches smaller than G * kChunkMin quads: chunks of exactly kChunkMin quads,
    the CTAs past the batch empty, and the cover still exact."""
    rng = np.random.default_rng(G + 5)
    for nq in (1, CHUNK_MIN - 1, CHUNK_MIN, CHUNK_MIN + 1, 3 * CHUNK_MIN, (G - 1) * CHUNK_MIN + 7):
        S, Sw, ranges = warp_ranges(nq, G)
        assert S == CHUNK_MIN
        live = [v for v, (lo, hi) in enumerate(ranges) if lo < hi]
        assert max(live) // K_WARPS == (nq - 1) // CHUNK_MIN          # the last CTA with work
        total = 4 * nq - int(rng.integers(0, 4))
        cuts = np.sort(rng.integers(0, total + 1, size=int(rng.integers(0, 40))))
        offsets = np.concatenate([[0], cuts, [total]]).astype(np.int64)
        emulate(offsets, 0, G, 4, 12)
        emulate(offsets, 0, G, 1, MAX_M)
