"""lookup_draft's per-stream scratch, against the oracle.

lookup_draft keeps the scan's result slots in one buffer per stream, made on the
first call outside stream capture and grown when a larger batch comes. Inside a
capture on a stream without a big-enough buffer, a call takes its scratch from
the library pool (graph memory nodes) instead.

Checked here:
- interleaved calls on two streams with different batches;
- a batch larger than the stream's buffer, then smaller ones again;
- a graph captured on a fresh stream (the pool path), and one captured after an
  eager call (the stream's buffer), each replayed several times;
- a graph replayed after a later, larger call replaced its stream's buffer (the
  old buffer stays allocated);
- lookup_draft_host, which stages its copy of the inputs, its outputs and the
  slots in the same per-stream buffer: interleaved with device calls on one
  stream (growing it), before and after graph capture, and from several threads
  on one shared stream, where each call holds the stream's lock while it enqueues
  its kernels.
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


@pytest.fixture(scope="module", autouse=True)
def _device_set_up():
    """The library's per-device set-up happens on its first call, which must come
    before any stream capture: one eager call on the default stream."""
    w = gen.make_workload("tiny")
    pkg.lookup_draft(torch.from_numpy(w.tokens).to(DEV), torch.from_numpy(w.offsets).to(DEV), 4, 12, 15)
    torch.cuda.synchronize()


def many_requests(B: int, seed: int):
    """B short requests over a 4-letter alphabet: more slots than a stream's first
    buffer (64 KiB, 8,192 slots) holds, so a call with it grows the buffer."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(0, 60, size=B)
    tokens = rng.integers(0, 4, size=int(lengths.sum())).astype(np.int32)
    return gen.Workload(name=f"many{B}", tokens=tokens, offsets=gen.offsets_from_lengths(lengths), min_m=4,
                        max_m=12, K=7, seed=seed, planted={})


class Batch:
    def __init__(self, name: str, seed: int):
        self.w = many_requests(12000, seed) if name == "many" else gen.make_workload(name, seed)
        self.t = torch.from_numpy(self.w.tokens).to(DEV)
        self.o = torch.from_numpy(self.w.offsets).to(DEV)
        self.want = oracle.lookup_draft(self.w.tokens, self.w.offsets, self.w.min_m, self.w.max_m, self.w.K,
                                        threads=8)

    def outputs(self):
        w = self.w
        return (torch.full((w.B, w.K), 7, dtype=torch.int32, device=DEV),
                torch.full((w.B,), 7, dtype=torch.int32, device=DEV),
                torch.full((w.B,), 7, dtype=torch.int32, device=DEV))

    def call(self, lib, out, stream):
        w = self.w
        d, ln, p = out
        rc = lib.lookup_draft(self.t.data_ptr(), self.o.data_ptr(), w.B, w.min_m, w.max_m, w.K, d.data_ptr(),
                              ln.data_ptr(), p.data_ptr(), stream.cuda_stream)
        assert rc == 0, (lib.lookup_draft_strerror(rc), lib.lookup_draft_last_cuda_error())

    def check(self, out, what: str):
        for name, g, e in zip(("draft", "len", "pos"), out, self.want[:3]):
            np.testing.assert_array_equal(g.cpu().numpy(), e, err_msg=f"{what}: {name}")


def test_two_streams_interleaved_with_growth():
    lib = pkg.load_library()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    small, big, other = Batch("tiny", 41), Batch("many", 42), Batch("recitation25k", 43)
    plan = [(small, s1), (other, s2), (big, s1), (small, s2), (other, s1), (big, s2), (small, s1)]
    outs = [(b, s, b.outputs()) for b, s in plan]
    torch.cuda.synchronize()                            # inputs and outputs made on the default stream
    for b, s, out in outs:
        with torch.cuda.stream(s):
            b.call(lib, out, s)
    torch.cuda.synchronize()
    for i, (b, _, out) in enumerate(outs):
        b.check(out, f"call {i}")


def test_growth_then_smaller_batches_on_one_stream():
    lib = pkg.load_library()
    s = torch.cuda.Stream()
    batches = [Batch("tiny", 44), Batch("ragged262k", 45), Batch("many", 46), Batch("chats", 47)]
    torch.cuda.synchronize()
    results = []
    with torch.cuda.stream(s):
        for b in batches + batches[::-1]:
            out = b.outputs()
            b.call(lib, out, s)
            results.append((b, out))
    torch.cuda.synchronize()
    for i, (b, out) in enumerate(results):
        b.check(out, f"call {i}")


@pytest.mark.parametrize("warm", [False, True])
def test_graph_on_fresh_and_warm_streams(warm):
    """warm=False: the capture finds no buffer for the stream and takes scratch from
    the pool; warm=True: an eager call first, so the graph uses the stream's buffer."""
    lib = pkg.load_library()
    s = torch.cuda.Stream()
    b1, b2 = Batch("recitation25k", 48), Batch("chats", 49)
    o1, o2 = b1.outputs(), b2.outputs()
    torch.cuda.synchronize()
    if warm:
        with torch.cuda.stream(s):
            b2.call(lib, o2, s)
        torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cs = torch.cuda.current_stream()
        for _ in range(3):
            b1.call(lib, o1, cs)
            b2.call(lib, o2, cs)
    for rep in range(3):
        for x in o1 + o2:
            x.fill_(7)
        g.replay()
        torch.cuda.synchronize()
        b1.check(o1, f"replay {rep}, first batch")
        b2.check(o2, f"replay {rep}, second batch")


def test_graph_replayed_after_its_buffer_was_replaced():
    lib = pkg.load_library()
    s = torch.cuda.Stream()
    small, big = Batch("tiny", 50), Batch("many", 51)
    o_small, o_big = small.outputs(), big.outputs()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        small.call(lib, o_small, s)                     # the stream's buffer, sized for the small batch
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        small.call(lib, o_small, torch.cuda.current_stream())
    with torch.cuda.stream(s):
        big.call(lib, o_big, s)                         # grows: a new buffer for this stream
    torch.cuda.synchronize()
    big.check(o_big, "larger batch")
    for x in o_small:
        x.fill_(7)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()                                      # still uses the first buffer, still allocated
    torch.cuda.synchronize()
    small.check(o_small, "graph replay after growth")


def test_threads_calling_on_their_own_and_shared_streams():
    """Four host threads (ctypes releases the GIL, so the library's host code runs
    concurrently): two on streams of their own, two sharing a third stream. Each
    call's outputs are its own, so every result can be checked afterwards."""
    import threading

    lib = pkg.load_library()
    own1, own2, shared = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    batches = [Batch("tiny", 60), Batch("many", 61), Batch("recitation25k", 62), Batch("chats", 63)]
    plan = [(own1, batches[0], batches[1]), (own2, batches[2], batches[3]),
            (shared, batches[0], batches[2]), (shared, batches[1], batches[3])]
    work = [[(b, b.outputs()) for _ in range(6) for b in (b1, b2)] for _, b1, b2 in plan]
    torch.cuda.synchronize()
    errors = []

    def run(stream, calls):
        try:
            for b, out in calls:
                b.call(lib, out, stream)
        except Exception as exc:  # surfaced below
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(s, calls)) for (s, _, _), calls in zip(plan, work)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i, calls in enumerate(work):
        for j, (b, out) in enumerate(calls):
            b.check(out, f"thread {i}, call {j}")


def test_per_thread_default_streams_get_their_own_scratch():
    """cudaStreamPerThread names a different stream in each thread: two threads
    passing that handle run concurrently and must not share one scratch buffer."""
    import threading

    lib = pkg.load_library()
    per_thread = 2                                      # the cudaStreamPerThread handle
    b1, b2 = Batch("recitation25k", 64), Batch("chats", 65)
    work = [[(b1, b1.outputs()) for _ in range(8)], [(b2, b2.outputs()) for _ in range(8)]]
    torch.cuda.synchronize()
    errors = []

    def run(calls):
        try:
            for b, (d, ln, p) in calls:
                w = b.w
                rc = lib.lookup_draft(b.t.data_ptr(), b.o.data_ptr(), w.B, w.min_m, w.max_m, w.K, d.data_ptr(),
                                      ln.data_ptr(), p.data_ptr(), per_thread)
                assert rc == 0, lib.lookup_draft_last_cuda_error()
            torch.cuda.synchronize()
        except Exception as exc:  # surfaced below
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(calls,)) for calls in work]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i, calls in enumerate(work):
        for j, (b, out) in enumerate(calls):
            b.check(out, f"thread {i}, call {j}")


class HostBatch:
    """A batch on host memory for lookup_draft_host: page-locked (read by the
    device's copy kernel, outputs written in place) or pageable (copy-engine
    transfers both ways)."""

    def __init__(self, name: str, seed: int, pinned: bool = True):
        self.w = many_requests(12000, seed) if name == "many" else gen.make_workload(name, seed)
        self.pinned = pinned
        self.t = self._host(torch.from_numpy(self.w.tokens))
        self.o = self._host(torch.from_numpy(self.w.offsets))
        self.want = oracle.lookup_draft(self.w.tokens, self.w.offsets, self.w.min_m, self.w.max_m, self.w.K,
                                        threads=8)

    def _host(self, x):
        return x.pin_memory() if self.pinned else x.clone()

    def outputs(self):
        w = self.w
        return tuple(self._host(torch.full(sh, 7, dtype=torch.int32)) for sh in ((w.B, w.K), (w.B,), (w.B,)))

    def call(self, lib, out, stream):
        w = self.w
        d, ln, p = out
        rc = lib.lookup_draft_host(self.t.data_ptr(), self.o.data_ptr(), w.B, w.min_m, w.max_m, w.K, d.data_ptr(),
                                   ln.data_ptr(), p.data_ptr(), stream.cuda_stream)
        assert rc == 0, (lib.lookup_draft_strerror(rc), lib.lookup_draft_last_cuda_error())

    def check(self, out, what: str):
        for name, g, e in zip(("draft", "len", "pos"), out, self.want[:3]):
            np.testing.assert_array_equal(g.numpy(), e, err_msg=f"{what}: {name}")


def test_host_and_device_calls_share_one_streams_buffer():
    """The host entry point copies its inputs into the stream's buffer, which the
    device calls before and after it on the same stream also use; each host call
    that needs more than the buffer holds grows it."""
    lib = pkg.load_library()
    s = torch.cuda.Stream()
    dev_calls = [Batch("tiny", 70), Batch("chats", 71), Batch("many", 72), Batch("tiny", 73)]
    host_calls = [HostBatch("recitation25k", 74), HostBatch("tiny", 75), HostBatch("ragged262k", 76),
                  HostBatch("chats", 77, pinned=False), HostBatch("periodic", 78)]
    dev_out = [b.outputs() for b in dev_calls]
    torch.cuda.synchronize()
    order = [("d", 0), ("h", 0), ("d", 1), ("h", 1), ("h", 2), ("d", 2), ("h", 3), ("d", 3), ("h", 4)]
    for kind, i in order:
        with torch.cuda.stream(s):
            if kind == "d":
                dev_calls[i].call(lib, dev_out[i], s)
            else:
                out = host_calls[i].outputs()
                host_calls[i].call(lib, out, s)              # synchronous: checked at once
                host_calls[i].check(out, f"host call {i}")
    torch.cuda.synchronize()
    for i, (b, out) in enumerate(zip(dev_calls, dev_out)):
        b.check(out, f"device call {i}")


@pytest.mark.parametrize("host_batch", ["tiny", "ragged262k"])
def test_graph_replayed_after_a_host_call_on_its_stream(host_batch):
    """A graph captured after an eager call uses the stream's buffer; a host call
    on that stream then reuses the buffer (tiny) or replaces it with a larger one
    (ragged262k). Replays that do not overlap the host call stay exact."""
    lib = pkg.load_library()
    s = torch.cuda.Stream()
    b = Batch("recitation25k", 80)
    h = HostBatch(host_batch, 81)
    o = b.outputs()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        b.call(lib, o, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.call(lib, o, torch.cuda.current_stream())
    ho = h.outputs()
    with torch.cuda.stream(s):
        h.call(lib, ho, s)
    h.check(ho, "host call")
    for rep in range(3):
        for x in o:
            x.fill_(7)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        b.check(o, f"replay {rep}")


def test_threads_mixing_host_and_device_calls_on_one_stream():
    """Four threads on ONE stream, each alternating device calls and host calls.
    Without the stream's lock, one thread's scan could land between another
    call's scan and fill (or its copy) on the shared stream and read that call's
    slots or staged tokens; with it every result is exact."""
    import threading

    lib = pkg.load_library()
    shared = torch.cuda.Stream()
    dev_b = [Batch("tiny", 90), Batch("recitation25k", 91), Batch("chats", 92), Batch("many", 93)]
    host_b = [HostBatch("periodic", 94), HostBatch("tiny", 95), HostBatch("recitation25k", 96),
              HostBatch("tiny", 97, pinned=False)]
    rounds = 8
    work = [[(dev_b[(i + k) % 4], dev_b[(i + k) % 4].outputs(), host_b[(i + 2 * k) % 4],
              host_b[(i + 2 * k) % 4].outputs()) for k in range(rounds)] for i in range(4)]
    torch.cuda.synchronize()
    errors = []

    def run(calls):
        try:
            for db, dout, hb, hout in calls:
                db.call(lib, dout, shared)
                hb.call(lib, hout, shared)
                hb.check(hout, "host call in a thread")
        except Exception as exc:  # surfaced below
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(calls,)) for calls in work]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i, calls in enumerate(work):
        for k, (db, dout, _, _) in enumerate(calls):
            db.check(dout, f"thread {i}, round {k}")
