"""The allocation-free entry point, lookup_draft_noalloc, against lookup_draft.

lookup_draft_noalloc serves callers that must not allocate device memory while
they draft (a serving loop whose GPU memory belongs to another allocator, a
process under a fixed device-memory budget): instead of taking the scan's
scratch from a memory pool it uses a fixed array compiled into the library.
Its results must be those of lookup_draft and of the CPU oracle, bit for bit,
including on later calls in a row, when the array still holds the earlier
calls' leftovers -- also over a batch with empty requests and offsets[0] > 0 at
the request indices an earlier call filled.

This file is collected last so that a run that stops at its first failure has
already run every other test; it also passes when run alone.
"""
from __future__ import annotations

import ctypes

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


def _batch(name: str, seed: int):
    w = gen.make_workload(name, seed)
    t = torch.from_numpy(w.tokens).to(DEV)
    o = torch.from_numpy(w.offsets).to(DEV)
    return w, t, o


def _holes(w, seed: int):
    """The workload with every third request emptied and 5 unowned tokens before
    offsets[0]: empty requests and a non-zero offsets[0] at the same indices as
    the full batch."""
    rng = np.random.default_rng(seed)
    lengths = np.diff(w.offsets)
    lengths[::3] = 0
    lead = 5
    keep = np.concatenate([w.tokens[w.offsets[r]:w.offsets[r + 1]] for r in range(w.B) if lengths[r]])
    tokens = np.concatenate([rng.integers(0, 100, lead), keep]).astype(np.int32)
    offsets = (gen.offsets_from_lengths(lengths) + lead).astype(np.int64)
    return gen.Workload(name=w.name + "-holes", tokens=tokens, offsets=offsets, min_m=w.min_m,
                        max_m=w.max_m, K=w.K, seed=w.seed, planted={})


def _noalloc(lib, w, t, o, stream):
    """lookup_draft_noalloc through the C ABI, into freshly made output tensors."""
    d = torch.full((w.B, w.K), 7, dtype=torch.int32, device=DEV)
    ln = torch.full((w.B,), 7, dtype=torch.int32, device=DEV)
    p = torch.full((w.B,), 7, dtype=torch.int32, device=DEV)
    rc = lib.lookup_draft_noalloc(t.data_ptr(), o.data_ptr(), w.B, w.min_m, w.max_m, w.K,
                                  d.data_ptr(), ln.data_ptr(), p.data_ptr(), stream)
    assert rc == 0, lib.lookup_draft_strerror(rc)
    return d, ln, p


def _expect_equal(got, ref, want, what):
    """Bit-exact against lookup_draft's outputs and against the oracle's."""
    for name, a, b, c in zip(("draft", "len", "pos"), got, ref, want):
        a = a.cpu().numpy()
        np.testing.assert_array_equal(a, b.cpu().numpy(), err_msg=f"{what}: {name} vs lookup_draft")
        np.testing.assert_array_equal(a, c, err_msg=f"{what}: {name} vs the oracle")


def test_noalloc_matches_lookup_draft_and_the_oracle_on_calls_in_a_row():
    lib = pkg.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    batches = [_batch("chats", 31),            # many short requests
               _batch("recitation25k", 32),    # few long requests: a different slot layout
               _batch("ragged262k", 33)]       # requests spanning many warp ranges
    w0 = batches[0][0]
    hw = _holes(w0, 34)
    batches.append((hw, torch.from_numpy(hw.tokens).to(DEV), torch.from_numpy(hw.offsets).to(DEV)))
    want = [oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8)[:3]
            for (w, _, _) in batches]
    ref = [pkg.lookup_draft(t, o, w.min_m, w.max_m, w.K) for (w, t, o) in batches]
    # the allocation-free calls back to back on one stream, no sync in between; the
    # last one reuses the first one's request indices with holes in the batch
    got = [_noalloc(lib, w, t, o, stream) for (w, t, o) in batches]
    torch.cuda.synchronize()
    for (w, _, _), g, r, x in zip(batches, got, ref, want):
        _expect_equal(g, r, x, w.name)
    # and again on the first batch, over the other calls' leftovers
    again = _noalloc(lib, *batches[0], stream)
    torch.cuda.synchronize()
    _expect_equal(again, ref[0], want[0], "chats again")


def test_noalloc_rejects_batches_beyond_its_scratch():
    lib = pkg.load_library()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = (1 << 16) - 16 * sms + 1          # one request more than the fixed array holds
    t = torch.zeros(B, dtype=torch.int32, device=DEV)
    o = torch.arange(B + 1, dtype=torch.int64, device=DEV)
    out = [torch.empty(n, dtype=torch.int32, device=DEV) for n in (B * 4, B, B)]
    rc = lib.lookup_draft_noalloc(t.data_ptr(), o.data_ptr(), B, 4, 12, 4,
                                  out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -3 and b"fixed scratch" in lib.lookup_draft_strerror(rc)
    # the largest batch it accepts still works
    B_ok = B - 1
    d, ln, p = pkg.lookup_draft_noalloc(t[:B_ok], o[:B_ok + 1], 1, 2, 1)
    torch.cuda.synchronize()
    assert int(ln.sum()) == 0 and bool((p == -1).all())
