"""The checked build of the drafting step (LOOKUP_DRAFT_CHECKED=1) on the GPU.

The checked library has the regular library's entry points.  Its scan and fill
kernels check the CSR offsets before they read a token through them, and check
every tile, suffix-table, token, scratch-slot, bulk-copy, offsets and output
index they compute.  A failed check sets a bit in the device's check word and
skips the access (include/lookup_draft.h, "Checked build").

- Valid batches. The outputs are bit-exact with the oracle and the check word
  stays 0: no check fires on correct indices. Covered: the five workloads, the
  hand-worked cases, and the shapes that reach every path of the kernels. Those
  are offsets in shared memory and in global memory, the rejection widths
  D = 1..4, unaligned token pointers with offsets[0] > 0 and empty requests,
  both fill kernels, K = 0 and the widest m range. Also the staged, host-buffer
  and allocation-free entry points, and the bounded waits running out.
- Invalid offsets. A decreasing pair, offsets[0] < 0, or a history of 2^31
  tokens: every request reports failure and the word holds exactly the offsets
  bit. Every offset of these batches points inside the tokens allocation, so no
  read could leave it even if a check were missing. The next valid call is
  exact again.
"""
from __future__ import annotations

import ctypes

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
OFFSETS_BIT = pkg.CHECK_BITS["offsets"]


@pytest.fixture(scope="module")
def lib():
    lib = pkg.load_checked_library()
    assert lib.lookup_draft_checked_build() == 1
    pkg.check_word(lib, clear=True)
    return lib


@pytest.fixture(autouse=True)
def _clean_word(lib):
    pkg.check_word(lib, clear=True)
    yield
    pkg.check_word(lib, clear=True)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def run_checked(lib, tokens: np.ndarray, offsets: np.ndarray, min_m, max_m, K, pad: int = 0):
    """lookup_draft_ex of the checked library; `pad` shifts the tokens pointer by
    that many int32 (and leaves that much room before the batch)."""
    B = offsets.size - 1
    buf = torch.zeros(tokens.size + pad + 4, dtype=torch.int32, device=DEV)
    if tokens.size:
        buf[pad:pad + tokens.size] = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).to(DEV)
    o = torch.from_numpy(np.ascontiguousarray(offsets, np.int64)).to(DEV)
    d = torch.full((B, K), 7, dtype=torch.int32, device=DEV)
    ln, p, m = (torch.full((B,), 7, dtype=torch.int32, device=DEV) for _ in range(3))
    rc = lib.lookup_draft_ex(buf.data_ptr() + 4 * pad, o.data_ptr(), B, min_m, max_m, K,
                             d.data_ptr() if K else None, ln.data_ptr(), p.data_ptr(), m.data_ptr(), _stream())
    assert rc == 0, lib.lookup_draft_strerror(rc)
    torch.cuda.synchronize()
    return d.cpu().numpy(), ln.cpu().numpy(), p.cpu().numpy(), m.cpu().numpy()


def assert_exact_and_clean(lib, tokens, offsets, min_m, max_m, K, pad=0):
    got = run_checked(lib, tokens, offsets, min_m, max_m, K, pad)
    want = oracle.lookup_draft(tokens, offsets, min_m, max_m, K, threads=8)
    for name, g, w in zip(("draft", "len", "pos", "mlen"), got, want):
        np.testing.assert_array_equal(g, w, err_msg=f"checked build: {name} differs from the oracle")
    assert pkg.check_word(lib) == 0


@pytest.mark.parametrize("seed", [None, 6, 7])
@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_workloads_exact_without_alarms(lib, name, seed):
    w = gen.make_workload(name, seed)
    assert_exact_and_clean(lib, w.tokens, w.offsets, w.min_m, w.max_m, w.K)


def test_hand_worked_cases(lib):
    for case in load_cases():
        d, ln, p, m = run_checked(lib, case.tokens, case.offsets, case.min_m, case.max_m, case.K)
        np.testing.assert_array_equal(m, case.expect_m, err_msg=case.name)
        np.testing.assert_array_equal(p, case.expect_pos, err_msg=case.name)
        np.testing.assert_array_equal(ln, case.expect_len, err_msg=case.name)
        np.testing.assert_array_equal(d, case.expect_draft, err_msg=case.name)
    assert pkg.check_word(lib) == 0


@pytest.mark.parametrize("min_m", [1, 2, 3, 4])
def test_every_rejection_width(lib, min_m):
    """D = min(min_m, 4) selects the kernel; dense matches over a 3-letter
    alphabet reach the extension, the partial and the two-request passes."""
    rng = np.random.default_rng(40 + min_m)
    lengths = rng.integers(0, 900, size=60)
    tokens = rng.integers(0, 3, size=int(lengths.sum())).astype(np.int32)
    assert_exact_and_clean(lib, tokens, gen.offsets_from_lengths(lengths), min_m, 12, 9)


@pytest.mark.parametrize("pad", [0, 1, 2, 3])
def test_unaligned_pointer_offset_base_and_empty_requests(lib, pad):
    rng = np.random.default_rng(pad)
    lengths = [0, 1, 4, 5, 0, 13, 12, 3, 100, 0, 6, 1, 2500, 0, 37]
    lead = 7
    body = rng.integers(0, 4, sum(lengths))
    tokens = np.concatenate([rng.integers(0, 3, lead), body]).astype(np.int32)
    assert_exact_and_clean(lib, tokens, gen.offsets_from_lengths(lengths) + lead, 4, 12, 15, pad=pad)


@pytest.mark.parametrize("B", [1024, 3000, 5000])
def test_lane_fill_and_offsets_in_global_memory(lib, B):
    """B >= 1024 takes the lane-per-request fill; B + 1 > 4097 keeps the offsets in
    global memory instead of shared memory."""
    rng = np.random.default_rng(B)
    lengths = rng.integers(0, 300, size=B)
    lengths[::97] = 20000                                  # a few requests spanning many scan warps
    tokens = rng.integers(0, 5, size=int(lengths.sum())).astype(np.int32)
    assert_exact_and_clean(lib, tokens, gen.offsets_from_lengths(lengths), 4, 12, 7)


@pytest.mark.parametrize("min_m,max_m,K", [(1, 32, 0), (32, 32, 64), (4, 12, 1)])
def test_m_and_k_extremes(lib, min_m, max_m, K):
    rng = np.random.default_rng(min_m + max_m + K)
    lengths = rng.integers(0, 3000, size=30)
    tokens = rng.integers(0, 2, size=int(lengths.sum())).astype(np.int32)
    assert_exact_and_clean(lib, tokens, gen.offsets_from_lengths(lengths), min_m, max_m, K)


def test_staged_host_and_noalloc_entry_points(lib):
    w = gen.make_workload("chats", 21)
    want = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8)
    t = torch.from_numpy(w.tokens).to(DEV)
    o = torch.from_numpy(w.offsets).to(DEV)
    B, K = w.B, w.K
    # staged, with a garbage workspace
    nbytes = lib.lookup_draft_workspace_bytes(B)
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device=DEV)
    d = torch.full((B, K), 7, dtype=torch.int32, device=DEV)
    ln, p = (torch.full((B,), 7, dtype=torch.int32, device=DEV) for _ in range(2))
    assert lib.lookup_draft_scan(t.data_ptr(), o.data_ptr(), B, w.min_m, w.max_m, ws.data_ptr(), nbytes,
                                 _stream()) == 0
    assert lib.lookup_draft_fill(t.data_ptr(), o.data_ptr(), B, w.min_m, w.max_m, K, ws.data_ptr(), nbytes,
                                 d.data_ptr(), ln.data_ptr(), p.data_ptr(), None, _stream()) == 0
    torch.cuda.synchronize()
    for g, e in zip((d, ln, p), want[:3]):
        np.testing.assert_array_equal(g.cpu().numpy(), e)
    # allocation-free
    d.fill_(7), ln.fill_(7), p.fill_(7)
    assert lib.lookup_draft_noalloc(t.data_ptr(), o.data_ptr(), B, w.min_m, w.max_m, K, d.data_ptr(),
                                    ln.data_ptr(), p.data_ptr(), _stream()) == 0
    torch.cuda.synchronize()
    for g, e in zip((d, ln, p), want[:3]):
        np.testing.assert_array_equal(g.cpu().numpy(), e)
    # host buffers: pageable, then page-locked
    for pinned in (False, True):
        tok = torch.from_numpy(w.tokens)
        off = torch.from_numpy(w.offsets)
        outs = [torch.full(s, 7, dtype=torch.int32) for s in ((B, K), (B,), (B,))]
        if pinned:
            tok, off = tok.pin_memory(), off.pin_memory()
            outs = [x.pin_memory() for x in outs]
        assert lib.lookup_draft_host(tok.data_ptr(), off.data_ptr(), B, w.min_m, w.max_m, K,
                                     *(x.data_ptr() for x in outs), _stream()) == 0
        for g, e in zip(outs, want[:3]):
            np.testing.assert_array_equal(g.numpy(), e)
    assert pkg.check_word(lib) == 0


def test_bounded_waits_running_out_raise_no_alarm(lib):
    """The failure path of the scan's bounded waits (drain, failure keys) stays
    inside its indices too."""
    w = gen.make_workload("ragged262k", 16)
    want = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8)
    try:
        lib.lookup_draft_set_wait_limit_ns(1)
        d, ln, p, m = run_checked(lib, w.tokens, w.offsets, w.min_m, w.max_m, w.K)
    finally:
        lib.lookup_draft_set_wait_limit_ns(0)
    ok = ln != pkg.LEN_FAILED
    np.testing.assert_array_equal(ln[ok], want[1][ok])
    np.testing.assert_array_equal(d[ok], want[0][ok])
    assert np.all(p[~ok] == -1) and np.all(d[~ok] == -1)
    assert pkg.check_word(lib) == 0
    assert_exact_and_clean(lib, w.tokens, w.offsets, w.min_m, w.max_m, w.K)


def _decreasing_pair(B: int, seed: int):
    """A batch of B short requests whose offsets decrease once in the middle;
    every offset stays inside [offsets[0], offsets[B]]."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 40, size=B)
    offsets = gen.offsets_from_lengths(lengths)
    r = B // 2
    offsets[r], offsets[r + 1] = offsets[r + 1], offsets[r]
    assert offsets[r] > offsets[r + 1]
    tokens = rng.integers(0, 3, size=int(offsets[-1])).astype(np.int32)
    return tokens, offsets


def _assert_all_failed(got, B, K):
    d, ln, p, m = got
    assert np.all(ln == pkg.LEN_FAILED) and np.all(p == -1) and np.all(m == 0)
    assert d.shape == (B, K) and np.all(d == -1)


@pytest.mark.parametrize("B", [3, 1100, 5000])
def test_decreasing_offsets_are_flagged(lib, B):
    """Both fill kernels (B < and >= 1024), offsets in shared and in global memory."""
    if B == 3:
        tokens = np.arange(1000, dtype=np.int32) % 7
        offsets = np.array([0, 300, 200, 1000], dtype=np.int64)
    else:
        tokens, offsets = _decreasing_pair(B, B)
    got = run_checked(lib, tokens, offsets, 4, 12, 15)
    _assert_all_failed(got, B, 15)
    assert pkg.check_word(lib, clear=True) == OFFSETS_BIT
    w = gen.make_workload("tiny", 3)
    assert_exact_and_clean(lib, w.tokens, w.offsets, w.min_m, w.max_m, w.K)


def test_negative_first_offset_is_flagged(lib):
    """offsets[0] = -4 with the tokens pointer 16 elements into its allocation, so
    even index -4 lies inside the allocation."""
    tokens = (np.arange(1100, dtype=np.int32) % 5)
    offsets = np.array([-4, 500, 1000], dtype=np.int64)
    got = run_checked(lib, tokens, offsets, 4, 12, 15, pad=16)
    _assert_all_failed(got, 2, 15)
    assert pkg.check_word(lib, clear=True) == OFFSETS_BIT


def test_history_of_2_pow_31_tokens_is_flagged(lib):
    """A request of 2^31 tokens (over the limit), in an allocation that holds them
    all, so the batch's range is inside the allocation either way."""
    n = (1 << 31) + 64
    buf = torch.empty(n, dtype=torch.int32, device=DEV)
    o = torch.tensor([0, 16, 16 + (1 << 31)], dtype=torch.int64, device=DEV)
    B, K = 2, 15
    d = torch.full((B, K), 7, dtype=torch.int32, device=DEV)
    ln, p, m = (torch.full((B,), 7, dtype=torch.int32, device=DEV) for _ in range(3))
    rc = lib.lookup_draft_ex(buf.data_ptr(), o.data_ptr(), B, 4, 12, K, d.data_ptr(), ln.data_ptr(), p.data_ptr(),
                             m.data_ptr(), _stream())
    assert rc == 0
    torch.cuda.synchronize()
    _assert_all_failed(tuple(x.cpu().numpy() for x in (d, ln, p, m)), B, K)
    assert pkg.check_word(lib, clear=True) == OFFSETS_BIT
    del buf
    torch.cuda.empty_cache()


def test_check_word_reads_and_clears(lib):
    out = ctypes.c_uint32(123)
    assert lib.lookup_draft_check_word(ctypes.byref(out), 1) == 0 and out.value == 0
    assert lib.lookup_draft_check_word(None, 0) == -1
    regular = pkg.load_library()
    assert regular.lookup_draft_checked_build() == 0
    assert regular.lookup_draft_check_word(ctypes.byref(out), 0) == 0 and out.value == 0


def _draft_plan(lib, t, o, B, md, committed, H, T, min_m=4, max_m=12):
    W = H + T
    out = [torch.full(s, 7, dtype=torch.int32, device=DEV) for s in ((B,), (B, W), (B,), (B, W), (B,), (B,))]
    state = torch.zeros((B, 3), dtype=torch.int32, device=DEV)
    rc = lib.lookup_draft_plan(t.data_ptr(), o.data_ptr(), B, min_m, max_m, md.data_ptr(), committed.data_ptr(), H, T,
                               8, 6, 2, 4, 1, 2, 3, state.data_ptr(), *(x.data_ptr() for x in out), _stream())
    assert rc == 0, lib.lookup_draft_strerror(rc)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in out] + [state.cpu().numpy()]


@pytest.mark.parametrize("name", ["recitation25k", "chats"])
def test_draft_plan_matches_the_regular_build_without_alarms(lib, name):
    regular = pkg.load_library()
    w = gen.make_workload(name, 24)
    t, o = torch.from_numpy(w.tokens).to(DEV), torch.from_numpy(w.offsets).to(DEV)
    H, T = 7, 8
    rng = np.random.default_rng(5)
    md = torch.from_numpy(rng.integers(0, 50, size=(w.B, H)).astype(np.int32)).to(DEV)
    committed = torch.from_numpy(rng.integers(1, H + T + 2, size=w.B).astype(np.int32)).to(DEV)
    got = _draft_plan(lib, t, o, w.B, md, committed, H, T)
    want = _draft_plan(regular, t, o, w.B, md, committed, H, T)
    for g, e in zip(got, want):
        np.testing.assert_array_equal(g, e)
    assert pkg.check_word(lib) == 0


def test_draft_plan_with_decreasing_offsets_plans_every_request_as_failed(lib):
    tokens, offsets = _decreasing_pair(1100, 77)
    B, H, T = offsets.size - 1, 3, 2
    t, o = torch.from_numpy(tokens).to(DEV), torch.from_numpy(offsets).to(DEV)
    md = torch.full((B, H), 5, dtype=torch.int32, device=DEV)
    committed = torch.ones(B, dtype=torch.int32, device=DEV)
    lng, blk, ln, pm, ml, dl, st = _draft_plan(lib, t, o, B, md, committed, H, T)
    assert np.all(dl == pkg.LEN_FAILED) and np.all(ml == 0)
    assert np.all(blk[:, :H] == 5) and np.all(blk[:, H:] == -1) and np.all(ln == H) and np.all(pm == 0)
    assert pkg.check_word(lib, clear=True) == OFFSETS_BIT
