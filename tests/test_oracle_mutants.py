"""The oracle's pins are strong enough to catch plausible mistakes.

Each case below plants one mistake in a copy of the oracle's C source (a wrong
loop direction, an off-by-one bound, a dropped comparison, a wrong sentinel ...),
compiles the copy with gcc into a temporary library, and runs the pins of
test_oracle_pins.py against it through the same ctypes wrapper.  Every mutant
must fail at least one pin.  The mistakes are planted on the CPU only; the real
oracle is never modified.
"""
from __future__ import annotations

import os
import subprocess

import numpy as np
import pytest

import gen
import oracle
from goldens import load_cases
from invariants import check_small

SRC = os.path.join(os.path.dirname(oracle.__file__), "lookup_oracle.c")
LOOP_SRC = os.path.join(os.path.dirname(oracle.__file__), "loop_oracle.c")
CTX_SRC = os.path.join(os.path.dirname(oracle.__file__), "ctx_oracle.c")

MUTANTS = {
    "oldest_first": ("for (int64_t p = L - m - 1; p >= 0; --p)",
                     "for (int64_t p = 0; p <= L - m - 1; ++p)"),
    "no_overlap": ("for (int64_t p = L - m - 1; p >= 0; --p)",
                   "for (int64_t p = L - 2 * m; p >= 0; --p)"),
    "suffix_counts_as_earlier": ("for (int64_t p = L - m - 1; p >= 0; --p)",
                                 "for (int64_t p = L - m; p >= 0; --p)"),
    "shortest_first": ("for (int64_t m = top; m >= (int64_t)min_m; --m)",
                       "for (int64_t m = (int64_t)min_m; m <= top; ++m)"),
    "min_m_excluded": ("for (int64_t m = top; m >= (int64_t)min_m; --m)",
                       "for (int64_t m = top; m > (int64_t)min_m; --m)"),
    "cap_too_low": ("top = L - 1;", "top = L - 2;"),
    "max_m_ignored": ("int64_t top = (int64_t)max_m;", "int64_t top = L - 1 + 0 * max_m;"),
    "first_token_skipped": ("if (t[a + i] != t[b + i])", "if (i > 0 && t[a + i] != t[b + i])"),
    "last_token_skipped": ("for (int64_t i = 0; i < n; ++i)", "for (int64_t i = 0; i + 1 < n; ++i)"),
    "no_self_extension": ("draft[j] = (src < L) ? t[src] : draft[src - L];",
                          "draft[j] = (src < L) ? t[src] : t[L - 1];"),
    "draft_off_by_one": ("int64_t src = p + m + j;", "int64_t src = p + m + j - 1;"),
    "wrong_position": ("out_pos[r] = (int32_t)p;", "out_pos[r] = (int32_t)(p + m);"),
    "wrong_sentinel": ("out_pos[r] = -1;", "out_pos[r] = 0;"),
    "short_draft_length": ("out_len[r] = K;", "out_len[r] = K - 1;"),
}


def _pins_fail(lib) -> list[str]:
    """Run the pins against a library; return the names of those that fail."""
    failed = []

    def run(tokens, offsets, min_m, max_m, K):
        return oracle.lookup_draft(tokens, offsets, min_m, max_m, K, lib=lib)

    for c in load_cases():
        d, ln, p, m = run(c.tokens, c.offsets, c.min_m, c.max_m, c.K)
        if not (np.array_equal(m, c.expect_m) and np.array_equal(p, c.expect_pos)
                and np.array_equal(ln, c.expect_len) and np.array_equal(d, c.expect_draft)):
            failed.append(f"golden:{c.name}")
    w = gen.make_workload("tiny")
    d, ln, p, m = run(w.tokens, w.offsets, w.min_m, w.max_m, w.K)
    for r, (s0, c) in w.planted.items():
        t = w.tokens[w.offsets[r]:w.offsets[r + 1]]
        if (m[r], p[r], ln[r]) != (12, s0 + c - 12, 15) or \
                not np.array_equal(d[r], t[s0 + c:s0 + c + 15]):
            failed.append("planted")
            break
    for dd in (1, 3, 7):
        a = np.arange(dd, dtype=np.int32) + 50
        L = dd + 12 + 5
        t = a[np.arange(L) % dd]
        d, ln, p, m = run(t, np.array([0, L], np.int64), 4, 12, 15)
        if (m[0], p[0]) != (12, L - 12 - dd) or \
                not np.array_equal(d[0], a[(L + np.arange(15)) % dd]):
            failed.append(f"periodic:{dd}")
    import itertools
    hists = [list(s) for L in range(0, 9) for s in itertools.product(range(2), repeat=L)]
    tokens = np.array([x for h in hists for x in h], dtype=np.int32)
    offsets = gen.offsets_from_lengths([len(h) for h in hists])
    for (min_m, max_m, K) in [(1, 3, 5), (2, 4, 1)]:
        d, ln, p, m = run(tokens, offsets, min_m, max_m, K)
        for r, h in enumerate(hists):
            if check_small(h, min_m, max_m, K, int(m[r]), int(p[r]), int(ln[r]), d[r]):
                failed.append(f"exhaustive:{min_m},{max_m}")
                break
    return failed


def test_unmutated_oracle_passes_the_pins():
    assert _pins_fail(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation target for {name} not found in the oracle"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated, encoding="utf-8")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", str(so_path),
                    str(c_path), LOOP_SRC, CTX_SRC], check=True)
    failed = _pins_fail(oracle.load(str(so_path)))
    assert failed, f"mutant {name} passed every pin"


# ------------------------------------------------------- loop-step oracle ----
LOOP_MUTANTS = {
    "replace_strict": ("if (m >= replace_min)", "if (m > replace_min)"),
    "agree_ignored": ("else if (m >= agree_min && agree)", "else if (m >= agree_min)"),
    "tail_threshold": ("int tail = is_long && m >= tail_min;", "int tail = is_long && m > tail_min;"),
    "tail_not_long": ("int tail = is_long && m >= tail_min;", "int tail = m >= tail_min;"),
    "no_sticky": ("st[2] -= 1;                              /* sticky exit: keep the long block */",
                  "st[0] = 0;"),
    "enter_at_once": ("if (st[1] >= enter_steps) {", "if (st[1] >= 1) {"),
    "full_ignores_long": ("int32_t full = (st[0] ? H + T : H) + 1;", "int32_t full = H + 1;"),
    "greedy_off_by_one": ("ok = block[a] == target[a];", "ok = block[a] == target[a + 1];"),
    "point_mass_ignored": ("qa = 1.0f;                       /* point mass on the lookup token */", "qa = qa;"),
    "no_bonus": ("commit[i] = i < a ? block[i] : (i == a ? target[a] : -1);",
                 "commit[i] = i < a ? block[i] : -1;"),
    "append_order": ("        for (int64_t i = offsets[r]; i < offsets[r + 1]; ++i)\n            out_tokens[pos++] = tokens[i];\n        for (int32_t j = 0; j < ncommit[r]; ++j)\n            out_tokens[pos++] = commit[(int64_t)r * W + j];",
                     "        for (int32_t j = 0; j < ncommit[r]; ++j)\n            out_tokens[pos++] = commit[(int64_t)r * W + j];\n        for (int64_t i = offsets[r]; i < offsets[r + 1]; ++i)\n            out_tokens[pos++] = tokens[i];"),
}


def _loop_pins_fail(lib) -> list[str]:
    import test_loop_oracle_pins as pins
    failed = []
    saved = oracle.load
    oracle.load = lambda path=None: lib
    try:
        for name in dir(pins):
            if name.startswith("test_"):
                try:
                    getattr(pins, name)()
                except (AssertionError, ValueError, Exception):  # noqa: B014 - any failure counts
                    failed.append(name)
    finally:
        oracle.load = saved
    return failed


def test_unmutated_loop_oracle_passes_its_pins():
    assert _loop_pins_fail(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(LOOP_MUTANTS))
def test_loop_mutant_is_caught(name, tmp_path):
    old, new = LOOP_MUTANTS[name]
    src = open(LOOP_SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation target for {name} not found in the loop oracle"
    c_path = tmp_path / "loop_mutant.c"
    so_path = tmp_path / "libloopmutant.so"
    c_path.write_text(src.replace(old, new, 1), encoding="utf-8")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", str(so_path), SRC, str(c_path), CTX_SRC],
                   check=True)
    assert _loop_pins_fail(oracle.load(str(so_path))), f"mutant {name} passed every pin"


# -------------------------------------------------- context-cache oracle ----

CTX_MUTANTS = {
    "tie_to_larger": ("if (b - a > best_c) {", "if (b - a >= best_c) {"),
    "share_strict": ("if (best_c * (int64_t)den[n - 1] >= (int64_t)num[n - 1] * total) {",
                     "if (best_c * (int64_t)den[n - 1] > (int64_t)num[n - 1] * total) {"),
    "last_occurrence_dropped": ("for (int64_t i = 0; i + n <= L - 1; ++i) {",
                                "for (int64_t i = 0; i + n <= L - 2; ++i) {"),
    "shortest_first": ("for (int32_t n = n_max; n >= n_min && !accepted; --n) {",
                       "for (int32_t n = n_min; n <= n_max && !accepted; ++n) {"),
    "drafts_not_in_context": ("g[k] = c < L ? t[c] : draft[c - L];", "g[k] = t[c < L ? c : L - 1];"),
    "min_count_ignored": ("if (total == 0 || total < min_count[n - 1])", "if (total == 0)"),
    "share_ignored": ("if (best_c * (int64_t)den[n - 1] >= (int64_t)num[n - 1] * total) {", "if (1) {"),
    "wrong_sentinel": ("draft[k] = -1;", "draft[k] = 0;"),
    "successor_off_by_one": ("succ[total++] = t[i + n];", "succ[total++] = t[i + n - 1];"),
}


def _ctx_pins_fail(lib) -> list[str]:
    import test_ctx_oracle_pins as pins
    failed = []
    saved = oracle.load
    oracle.load = lambda path=None: lib
    try:
        for name in dir(pins):
            if name.startswith("test_"):
                fn = getattr(pins, name)
                params = getattr(fn, "pytestmark", [])
                cases = [{}]
                for mark in params:
                    if mark.name == "parametrize":
                        argname, values = mark.args
                        cases = [{argname: v} for v in values]
                for kw in cases:
                    try:
                        fn(**kw)
                    except (AssertionError, ValueError, Exception):  # noqa: B014 - any failure counts
                        failed.append(f"{name}{kw}")
    finally:
        oracle.load = saved
    return failed


def test_unmutated_ctx_oracle_passes_its_pins():
    assert _ctx_pins_fail(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(CTX_MUTANTS))
def test_ctx_mutant_is_caught(name, tmp_path):
    old, new = CTX_MUTANTS[name]
    src = open(CTX_SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation target for {name} not found in the context-cache oracle"
    c_path = tmp_path / "ctx_mutant.c"
    so_path = tmp_path / "libctxmutant.so"
    c_path.write_text(src.replace(old, new, 1), encoding="utf-8")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", str(so_path), SRC, LOOP_SRC, str(c_path)],
                   check=True)
    assert _ctx_pins_fail(oracle.load(str(so_path))), f"mutant {name} passed every pin"


# ------------------------------------------------------ controller oracle ----
POLICY_SRC = os.path.join(os.path.dirname(oracle.__file__), "policy_oracle.c")

POLICY_MUTANTS = {
    "edge_strict": ("if (m >= edge[i])", "if (m > edge[i])"),
    "margin_ignored": ("benefit_lookup > (1.0f + margin) * benefit_model", "benefit_lookup > benefit_model"),
    "tie_goes_to_lookup": ("benefit_lookup > (1.0f + margin) * benefit_model",
                           "benefit_lookup >= (1.0f + margin) * benefit_model"),
    "no_bonus_token": ("float sum = 1.0f;", "float sum = 0.0f;"),
    "weights_swapped": ("const float kept = (1.0f - alpha) * acc[slot];", "const float kept = alpha * acc[slot];"),
    "update_wrong_bucket": ("const int32_t slot = last == 2 ? prev[1] : 4;",
                            "const int32_t slot = last == 2 ? bucket_of(m, edge) : 4;"),
    "model_update_to_lookup": ("const int32_t slot = last == 2 ? prev[1] : 4;",
                               "const int32_t slot = last == 2 ? prev[1] : 0;"),
    "no_plain_fallback": ("if (!(best > benefit_plain))", "if (0)"),
    "no_clamp": ("if (a > n)\n            a = n;", ""),
    "lookup_without_match": ("const int lookup_available = m > 0;", "const int lookup_available = 1;"),
}


def _policy_pins_fail(lib) -> list[str]:
    import test_policy_oracle_pins as pins
    failed = []
    saved = oracle.load
    oracle.load = lambda path=None: lib
    try:
        for name in dir(pins):
            if name.startswith("test_"):
                try:
                    getattr(pins, name)()
                except (AssertionError, ValueError, Exception):  # noqa: B014 - any failure counts
                    failed.append(name)
    finally:
        oracle.load = saved
    return failed


def test_unmutated_policy_oracle_passes_its_pins():
    assert _policy_pins_fail(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(POLICY_MUTANTS))
def test_policy_mutant_is_caught(name, tmp_path):
    old, new = POLICY_MUTANTS[name]
    src = open(POLICY_SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation target for {name} not found in the controller oracle"
    c_path = tmp_path / "policy_mutant.c"
    so_path = tmp_path / "libpolicymutant.so"
    c_path.write_text(src.replace(old, new, 1), encoding="utf-8")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", str(so_path), SRC, LOOP_SRC, CTX_SRC,
                    str(c_path)], check=True)
    assert _policy_pins_fail(oracle.load(str(so_path))), f"mutant {name} passed every pin"
