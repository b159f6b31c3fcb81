"""Seeded synthetic inputs for prompt-lookup drafting.

This module only draws token histories; it holds none of the drafting
arithmetic, so both the CUDA path's tests and the CPU oracle take their inputs
from here without sharing any of the method's code.

A batch is a CSR pair: ``tokens`` (int32, the histories concatenated) and
``offsets`` (int64, B+1 entries, request r is tokens[offsets[r]:offsets[r+1]]).

The five named workloads stand in for the workloads of the pages, whose corpora
are not available here: HyperQwen's 25k-token verbatim recitation and short
chats, and list-like periodic text (HyperQwen lookup-drafting article,
sections "先看效果" and "第1步").  Every random choice goes through numpy's
PCG64 generator seeded with (seed, workload index).
"""
from __future__ import annotations

import dataclasses
import functools

import numpy as np

VOCAB_QWEN = 151936   # vocabulary size of the Qwen tokenizer the pages' models use


@dataclasses.dataclass
class Workload:
    name: str
    tokens: np.ndarray          # int32 [offsets[-1]]
    offsets: np.ndarray         # int64 [B + 1]
    min_m: int
    max_m: int
    K: int
    seed: int
    planted: dict               # request -> (source start s0, copy length c)

    @property
    def B(self) -> int:
        return int(self.offsets.shape[0]) - 1

    @property
    def total_tokens(self) -> int:
        return int(self.offsets[-1] - self.offsets[0])

    @property
    def history_bytes(self) -> int:
        return 4 * self.total_tokens


WORKLOADS = ("tiny", "recitation25k", "periodic", "ragged262k", "chats")
DEFAULT_SEED = {"tiny": 1, "recitation25k": 2, "periodic": 3, "ragged262k": 4, "chats": 5}

DESCRIPTION = {
    "tiny": "B=8, L=4096, uniform vocab 32000; 4 requests end in a 64-token copy of a "
            "span starting in [500,3000); min_m=4 max_m=12 K=15",
    "recitation25k": "B=64, L=25000, Zipf(1.1) over vocab 151936 (permuted); 30% of requests "
                     "end 1-2000 tokens into a copy of an earlier 2000-token span; "
                     "min_m=4 max_m=12 K=15",
    "periodic": "B=64, L=8192, runs of random periods 3-40 (run length 50-500), 5% uniform "
                "mutations, vocab 151936; min_m=4 max_m=12 K=7",
    "ragged262k": "B=256, L log-uniform in [512, 262144], Zipf(1.1); 20% end in a copy of an "
                  "earlier 1-4k span; min_m=4 max_m=12 K=15",
    "chats": "B=4096, L=2048, Zipf(1.2); 10% end in a 32-256-token copy of an earlier span; "
             "min_m=4 max_m=12 K=7",
}


def rng_for(seed: int, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


@functools.lru_cache(maxsize=8)
def _zipf_cdf(vocab: int, s: float) -> np.ndarray:
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    w = ranks ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    return cdf


def zipf_tokens(rng: np.random.Generator, n: int, vocab: int, s: float,
                perm: np.ndarray) -> np.ndarray:
    """n tokens with P(rank k) proportional to k^-s, rank k mapped to token perm[k-1]."""
    cdf = _zipf_cdf(vocab, s)
    u = rng.random(n)
    idx = np.searchsorted(cdf, u, side="right")
    np.minimum(idx, vocab - 1, out=idx)
    return perm[idx].astype(np.int32)


def uniform_tokens(rng: np.random.Generator, n: int, vocab: int) -> np.ndarray:
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def offsets_from_lengths(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)


def plant_copy(hist: np.ndarray, s0: int, c: int) -> None:
    """Make the history end in a verbatim copy of hist[s0 : s0 + c] (in place)."""
    L = hist.shape[0]
    assert 0 <= s0 and s0 + c <= L - c, (s0, c, L)
    hist[L - c:] = hist[s0:s0 + c]


def _choose(rng: np.random.Generator, B: int, frac: float) -> np.ndarray:
    n = int(round(frac * B))
    return np.sort(rng.permutation(B)[:n])


def make_workload(name: str, seed: int | None = None, length: int | None = None) -> Workload:
    """The named workload's batch.  ``length`` (recitation25k only, >= 4001)
    replaces the 25,000-token history length, with every other draw of the
    recipe unchanged; the workload is then named recitation_L<length>."""
    if name not in WORKLOADS:
        raise KeyError(f"unknown workload {name!r}; known: {WORKLOADS}")
    if length is not None and (name != "recitation25k" or int(length) < 4001):
        raise ValueError("length applies to recitation25k only, and must be at least 4001")
    seed = DEFAULT_SEED[name] if seed is None else int(seed)
    rng = rng_for(seed, WORKLOADS.index(name))
    planted: dict = {}

    if name == "tiny":
        B, L = 8, 4096
        tokens = uniform_tokens(rng, B * L, 32000)
        offsets = offsets_from_lengths([L] * B)
        for r in _choose(rng, B, 0.5):
            s0 = int(rng.integers(500, 3000))
            plant_copy(tokens[r * L:(r + 1) * L], s0, 64)
            planted[int(r)] = (s0, 64)
        return Workload(name, tokens, offsets, 4, 12, 15, seed, planted)

    if name == "periodic":
        B, L = 64, 8192
        rows = []
        for _ in range(B):
            parts, n = [], 0
            while n < L:
                d = int(rng.integers(3, 41))
                run = int(rng.integers(50, 501))
                pattern = uniform_tokens(rng, d, VOCAB_QWEN)
                parts.append(np.resize(pattern, run))
                n += run
            h = np.concatenate(parts)[:L].copy()
            flip = rng.random(L) < 0.05
            h[flip] = uniform_tokens(rng, int(flip.sum()), VOCAB_QWEN)
            rows.append(h)
        tokens = np.concatenate(rows).astype(np.int32)
        offsets = offsets_from_lengths([L] * B)
        return Workload(name, tokens, offsets, 4, 12, 7, seed, planted)

    perm = rng.permutation(VOCAB_QWEN).astype(np.int64)
    if name == "recitation25k":
        B, s, frac = 64, 1.1, 0.3
        lengths = np.full(B, 25000 if length is None else int(length), dtype=np.int64)
        K = 15
        if length is not None:
            name = f"recitation_L{int(length)}"
    elif name == "ragged262k":
        B, s, frac = 256, 1.1, 0.2
        lengths = np.floor(np.exp(rng.uniform(np.log(512), np.log(262144), size=B))).astype(np.int64)
        K = 15
    else:  # chats
        B, s, frac = 4096, 1.2, 0.1
        lengths = np.full(B, 2048, dtype=np.int64)
        K = 7
    offsets = offsets_from_lengths(lengths)
    tokens = zipf_tokens(rng, int(offsets[-1]), VOCAB_QWEN, s, perm)
    for r in _choose(rng, B, frac):
        r = int(r)
        L = int(lengths[r])
        if name.startswith("recitation"):
            span = 2000
            c = int(rng.integers(1, 2001))
            s0 = int(rng.integers(0, L - c - span + 1))
        elif name == "ragged262k":
            c = int(rng.integers(1024, 4097))
            c = min(c, L // 2 - 1)
            s0 = int(rng.integers(0, L - 2 * c + 1))
        else:
            c = int(rng.integers(32, 257))
            s0 = int(rng.integers(0, L - 2 * c + 1))
        h = tokens[offsets[r]:offsets[r + 1]]
        plant_copy(h, s0, c)
        planted[r] = (s0, c)
    return Workload(name, tokens, offsets, 4, 12, K, seed, planted)


# ----------------------------------------------------------- loop-step inputs ----
# Random inputs for the decode-loop steps (fusion, scheduling, verification,
# append).  As above, only draws: no rule of the method is applied here.  Values
# are concentrated where the rules have their thresholds (match lengths 3..8,
# commit counts near a full short or long block, exact ties in the sampled
# acceptance test) so that every branch is taken often.

def loop_fuse_inputs(B: int, K: int, H: int, T: int, agree_n: int, seed: int, vocab: int = 50):
    """(lookup_draft [B,K], lookup_mlen [B], model_draft [B,H], long_block [B])."""
    rng = rng_for(seed, 101)
    ld = rng.integers(0, vocab, size=(B, K), dtype=np.int64).astype(np.int32)
    special = np.array([0, 3, 4, 5, 6, 7, 8, 9, 12], np.int32)
    m = np.where(rng.random(B) < 0.7, special[rng.integers(0, special.size, size=B)],
                 rng.integers(0, 17, size=B)).astype(np.int32)
    md = rng.integers(0, vocab, size=(B, H), dtype=np.int64).astype(np.int32)
    copy = rng.random(B) < 0.5                       # the model proposes the lookup's head ...
    md[copy] = ld[copy, :H]
    if agree_n > 0:                                  # ... sometimes with one agreement token changed
        bump = copy & (rng.random(B) < 0.3)
        col = rng.integers(0, agree_n, size=B)
        md[bump, col[bump]] += 1
    long_block = (rng.random(B) < 0.5).astype(np.int32)
    return ld, m, md, long_block


def loop_schedule_trace(B: int, steps: int, H: int, T: int, seed: int):
    """(lookup_mlen [steps,B], committed [steps,B]): each request switches at random
    between copying (long matches, nearly full commits) and free text."""
    rng = rng_for(seed, 102)
    copying = rng.random(B) < 0.5
    mlen = np.empty((steps, B), np.int32)
    committed = np.empty((steps, B), np.int32)
    for s in range(steps):
        flip = rng.random(B) < 0.15
        copying = np.where(flip, ~copying, copying)
        m_copy = rng.integers(3, 13, size=B)
        m_free = np.where(rng.random(B) < 0.6, 0, rng.integers(0, 7, size=B))
        mlen[s] = np.where(copying, m_copy, m_free)
        near = np.array([H - 1, H, H + 1, H + T - 1, H + T, H + T + 1])
        c_copy = near[rng.integers(0, near.size, size=B)]
        c_free = rng.integers(1, H + T + 2, size=B)
        committed[s] = np.maximum(np.where(copying, c_copy, c_free), 1)
    return mlen, committed


def loop_verify_inputs(B: int, P: int, seed: int, vocab: int = 50):
    """(block [B,P], len [B], target [B,P+1], probs, qprobs, point_mass, u) with the
    target agreeing with the block on a random prefix, and exact ties u*q == p."""
    rng = rng_for(seed, 103)
    block = rng.integers(0, vocab, size=(B, P), dtype=np.int64).astype(np.int32)
    length = rng.integers(0, P + 1, size=B).astype(np.int32)
    full = rng.random(B) < 0.3
    length[full] = P
    target = rng.integers(0, vocab, size=(B, P + 1), dtype=np.int64).astype(np.int32)
    first_diff = rng.integers(0, P + 1, size=B)
    first_diff[rng.random(B) < 0.3] = P
    for r in range(B):
        f = int(first_diff[r])
        target[r, :f] = block[r, :f]
        if f < P:
            target[r, f] = block[r, f] + 1
    probs = rng.random((B, P), dtype=np.float32)
    qprobs = (1.0 - rng.random((B, P), dtype=np.float32)).astype(np.float32)   # (0, 1]
    u = rng.random((B, P), dtype=np.float32)
    tie = rng.random((B, P)) < 0.05                  # u * 1 == p exactly
    qprobs[tie] = 1.0
    probs[tie] = u[tie]
    half = (~tie) & (rng.random((B, P)) < 0.05)      # u * 0.5 == p exactly
    qprobs[half] = 0.5
    probs[half] = u[half] * np.float32(0.5)
    easy = rng.random(B) < 0.4                       # long accepted runs
    probs[easy] = np.float32(0.999)
    point_mass = (rng.random((B, P)) < 0.5).astype(np.int32)
    return block, length, target, probs, qprobs, point_mass, u


def loop_append_inputs(B: int, W: int, seed: int, vocab: int = VOCAB_QWEN):
    """(commit [B,W], ncommit [B]) with counts in [0, W]."""
    rng = rng_for(seed, 104)
    commit = rng.integers(0, vocab, size=(B, W), dtype=np.int64).astype(np.int32)
    ncommit = rng.integers(0, W + 1, size=B).astype(np.int32)
    return commit, ncommit


# ------------------------------------------------------------- slab layout ----
def slabs_from_batch(tokens: np.ndarray, offsets: np.ndarray, spare: int, seed: int, gap_max: int = 40,
                     fill: int = -5):
    """Lay a CSR batch out as capacity-padded slabs: request r's history at
    slab_tokens[base[r] : base[r] + len[r]], room for `spare` more tokens after
    it, then a random gap.  Everything outside the histories holds `fill`.
    Returns (slab_tokens int32, base int64 [B], len int32 [B], cap int32 [B])."""
    rng = rng_for(seed, 105)
    B = int(offsets.shape[0]) - 1
    lens = (offsets[1:] - offsets[:-1]).astype(np.int64)
    caps = lens + int(spare)
    gaps = rng.integers(0, gap_max + 1, size=B)
    base = np.zeros(B, np.int64)
    pos = int(rng.integers(0, gap_max + 1))
    for r in range(B):
        base[r] = pos
        pos += int(caps[r] + gaps[r])
    out = np.full(pos + 1, fill, np.int32)
    for r in range(B):
        out[base[r]:base[r] + lens[r]] = tokens[offsets[r]:offsets[r + 1]]
    return out, base, lens.astype(np.int32), caps.astype(np.int32)


def csr_of_slabs(slab_tokens: np.ndarray, base: np.ndarray, length: np.ndarray):
    """The CSR batch (tokens, offsets) holding the slabs' histories."""
    parts = [slab_tokens[int(b):int(b) + int(n)] for b, n in zip(base, length)]
    offsets = offsets_from_lengths([int(n) for n in length])
    tokens = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
    return tokens, offsets
