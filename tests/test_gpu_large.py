"""Batches larger than 2^31 tokens, and larger than 2^31 quads: the 64-bit offset
arithmetic end to end, and the scan's and the fill's 64-bit partition path.

A history of 2^31 - 1000 tokens, built as x_i = (i * a) mod P for a prime P, so
its only repeated 12-grams are exactly P apart; a short request with a planted
copy; and a request that starts beyond 2^31 tokens, also with a planted copy.
The draft step is compared with the oracle on every request; the CSR append
is compared on its boundaries and on a million sampled positions (the expected
token of a position follows from the boundaries alone).
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle

torch = pytest.importorskip("torch")
pkg = pytest.importorskip("prompt_lookup_speculative_gb300")

pytestmark = pytest.mark.gpu

P = 1_000_003
A = 2_654_435_761 % P


def big_batch():
    L0 = (1 << 31) - 1000
    rng = gen.rng_for(31, 71)
    small = rng.integers(0, 1 << 20, size=5000).astype(np.int32)
    small[-12:] = small[1000:1012]                       # its only 12-gram repeat: p = 1000
    far = rng.integers(0, 1 << 20, size=70_000).astype(np.int32)
    far[-15:] = far[20_000:20_015]                       # p = 20_003 (the last 12 of the 15)
    total = L0 + small.size + far.size
    tokens = np.empty(total, dtype=np.int32)
    step = 1 << 26
    for s in range(0, L0, step):                         # x_i = (i * A) mod P, in chunks
        e = min(s + step, L0)
        tokens[s:e] = (np.arange(s, e, dtype=np.int64) * A % P).astype(np.int32)
    tokens[L0:L0 + small.size] = small
    tokens[L0 + small.size:] = far
    offsets = np.array([0, L0, L0 + small.size, total], dtype=np.int64)
    return tokens, offsets


@pytest.fixture(scope="module")
def batch():
    tokens, offsets = big_batch()
    dev_tokens = torch.from_numpy(tokens).cuda()
    dev_offsets = torch.from_numpy(offsets).cuda()
    return tokens, offsets, dev_tokens, dev_offsets


def test_draft_beyond_2_31_tokens(batch):
    tokens, offsets, t, o = batch
    assert offsets[-1] > (1 << 31) and offsets[2] > (1 << 31)
    d, ln, pos, m = pkg.lookup_draft_ex(t, o, 4, 12, 15)
    torch.cuda.synchronize()
    od, oln, opos, om = oracle.lookup_draft(tokens, offsets, 4, 12, 15, threads=3)
    np.testing.assert_array_equal(m.cpu().numpy(), om)
    np.testing.assert_array_equal(pos.cpu().numpy(), opos)
    np.testing.assert_array_equal(ln.cpu().numpy(), oln)
    np.testing.assert_array_equal(d.cpu().numpy(), od)
    L0 = int(offsets[1])
    assert (int(om[0]), int(opos[0])) == (12, L0 - 12 - P)
    assert (int(om[1]), int(opos[1])) == (12, 1000)
    assert (int(om[2]), int(opos[2])) == (12, 20_003)


def test_append_beyond_2_31_tokens(batch):
    tokens, offsets, t, o = batch
    B, W = 3, 16
    commit = np.arange(B * W, dtype=np.int32).reshape(B, W) + 7_000_000
    ncommit = np.array([16, 0, 9], np.int32)
    out_t, out_o = pkg.lookup_append(t, o, torch.from_numpy(commit).cuda(), torch.from_numpy(ncommit).cuda())
    torch.cuda.synchronize()
    lens = np.diff(offsets)
    want_o = np.concatenate([[0], np.cumsum(lens + ncommit)])
    np.testing.assert_array_equal(out_o.cpu().numpy(), want_o)
    # positions: every request's first and last 64 and its commit, and a million random ones
    rng = gen.rng_for(3, 72)
    xs = [rng.integers(0, int(want_o[-1]), size=1_000_000)]
    for r in range(B):
        xs.append(np.arange(want_o[r], min(want_o[r] + 64, want_o[r + 1])))
        xs.append(np.arange(max(want_o[r + 1] - 64 - W, want_o[r]), want_o[r + 1]))
    xs = np.unique(np.concatenate(xs)).astype(np.int64)
    got = out_t[torch.from_numpy(xs).cuda()].cpu().numpy()
    r = np.searchsorted(want_o, xs, side="right") - 1
    i = xs - want_o[r]
    in_hist = i < lens[r]
    want = np.where(in_hist, tokens[np.minimum(offsets[r] + i, offsets[-1] - 1)],
                    commit[r, np.clip(i - lens[r], 0, W - 1)])
    np.testing.assert_array_equal(got, want)


def test_draft_beyond_2_31_quads():
    """A batch of more than 2^31 quads (about 36 GB of int32 history), which takes
    the scan's and the fill's 64-bit partition arithmetic.  Five requests of about
    1.8e9 tokens, request i built as x_j = (j * A_i) mod P_i on the device: its
    only repeated 12-grams are exactly P_i apart, so its most recent 12-token match
    is at p = L - 12 - P_i and the draft continues the period."""
    props = torch.cuda.get_device_properties(0)
    Ls = [1_800_000_000 + 7 * i for i in range(5)]
    total = sum(Ls)
    need = total * 4 + (2 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free on {props.name}")
    assert total // 4 >= (1 << 31)
    primes = [999_983, 1_000_003, 1_000_033, 999_979, 1_000_037]
    t = torch.empty(total, dtype=torch.int32, device="cuda")
    step = 1 << 27
    base = 0
    for L, P in zip(Ls, primes):
        A = 2_654_435_761 % P
        for s in range(0, L, step):
            e = min(s + step, L)
            t[base + s:base + e] = (torch.arange(s, e, dtype=torch.int64, device="cuda") * A % P).to(torch.int32)
        base += L
    offsets = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int64)
    o = torch.from_numpy(offsets).cuda()
    K = 15
    d, ln, pos, m = pkg.lookup_draft_ex(t, o, 4, 12, K)
    torch.cuda.synchronize()
    d, ln, pos, m = d.cpu().numpy(), ln.cpu().numpy(), pos.cpu().numpy(), m.cpu().numpy()
    del t
    torch.cuda.empty_cache()
    for i, (L, P) in enumerate(zip(Ls, primes)):
        A = 2_654_435_761 % P
        p = L - 12 - P
        assert (int(ln[i]), int(m[i]), int(pos[i])) == (K, 12, p), i
        want = [((p + 12 + j) * A) % P for j in range(K)]      # t[p + m + j], inside the history
        np.testing.assert_array_equal(d[i], np.array(want, dtype=np.int32))
