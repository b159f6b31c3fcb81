"""The allocation-free entry point, lookup_draft_noalloc, against lookup_draft.

lookup_draft_noalloc serves callers that must not allocate device memory while
they draft (a serving loop whose GPU memory belongs to another allocator, a
process under a fixed device-memory budget): instead of taking the scan's
scratch from a memory pool it uses a fixed array compiled into the library.
Its results must be those of lookup_draft, bit for bit, including on the second
of two calls in a row, when the array still holds the first call's leftovers.

This file is collected last so that a run that stops at its first failure has
already run every other test; it also passes when run alone.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import gen

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


def _noalloc(lib, w, t, o, stream):
    """lookup_draft_noalloc through the C ABI, into freshly made output tensors."""
    d = torch.full((w.B, w.K), 7, dtype=torch.int32, device=DEV)
    ln = torch.full((w.B,), 7, dtype=torch.int32, device=DEV)
    p = torch.full((w.B,), 7, dtype=torch.int32, device=DEV)
    rc = lib.lookup_draft_noalloc(t.data_ptr(), o.data_ptr(), w.B, w.min_m, w.max_m, w.K,
                                  d.data_ptr(), ln.data_ptr(), p.data_ptr(), stream)
    assert rc == 0, lib.lookup_draft_strerror(rc)
    return d, ln, p


def test_noalloc_matches_lookup_draft_on_two_calls_in_a_row():
    lib = pkg.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    first = _batch("chats", 31)            # many short requests
    second = _batch("recitation25k", 32)   # few long requests: a different slot layout
    ref = [pkg.lookup_draft(t, o, w.min_m, w.max_m, w.K) for (w, t, o) in (first, second)]
    # the two allocation-free calls back to back on one stream, no sync in between
    got = [_noalloc(lib, w, t, o, stream) for (w, t, o) in (first, second)]
    torch.cuda.synchronize()
    for g, r in zip(got, ref):
        for a, b in zip(g, r):
            np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())
    # and again on the first batch, over the second call's leftovers
    again = _noalloc(lib, *first, stream)
    torch.cuda.synchronize()
    for a, b in zip(again, ref[0]):
        np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())


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
