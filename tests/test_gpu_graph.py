"""The draft step as the benchmark runs it: calls captured in one CUDA graph, back
to back on one stream (programmatic dependent launch between the scan and fill
kernels and between consecutive steps), over several device copies of a
workload drawn with different seeds, and replayed.  Every step's outputs must
equal the oracle's, bit for bit, on every replay.
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
COPIES = 3


@pytest.mark.parametrize("name", gen.WORKLOADS)
def test_graph_captured_steps_match_the_oracle(name):
    ws = [gen.make_workload(name, gen.DEFAULT_SEED[name] + 100 + i) for i in range(COPIES)]
    toks = [torch.from_numpy(w.tokens).to(DEV) for w in ws]
    offs = [torch.from_numpy(w.offsets).to(DEV) for w in ws]
    outs = [(torch.empty((w.B, w.K), dtype=torch.int32, device=DEV),
             torch.empty(w.B, dtype=torch.int32, device=DEV),
             torch.empty(w.B, dtype=torch.int32, device=DEV),
             torch.empty(w.B, dtype=torch.int32, device=DEV)) for w in ws]
    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):          # first calls outside the capture: device set-up
        for i, w in enumerate(ws):
            pkg.lookup_draft_ex(toks[i], offs[i], w.min_m, w.max_m, w.K, out=outs[i], stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(2):                   # each copy twice: steps follow steps of other batches
            for i, w in enumerate(ws):
                pkg.lookup_draft_ex(toks[i], offs[i], w.min_m, w.max_m, w.K, out=outs[i],
                                    stream=torch.cuda.current_stream())
    wants = [oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=8) for w in ws]
    for replay in range(2):
        for o in outs:
            for t in o:
                t.fill_(-77)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for i, w in enumerate(ws):
            for label, got, want in zip(("draft", "len", "pos", "mlen"), outs[i], wants[i]):
                np.testing.assert_array_equal(got.cpu().numpy(), want,
                                              err_msg=f"{name} copy {i} replay {replay}: {label}")
