"""Loader for the hand-worked drafting fixtures in tests/golden/."""
from __future__ import annotations

import dataclasses
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@dataclasses.dataclass
class GoldenCase:
    name: str
    tokens: np.ndarray
    offsets: np.ndarray
    min_m: int
    max_m: int
    K: int
    expect_m: np.ndarray
    expect_pos: np.ndarray
    expect_len: np.ndarray
    expect_draft: np.ndarray      # [B, K]


def _ints(text: str) -> list[int]:
    return [int(x) for x in text.split()]


def load_cases(filename: str = "hand_worked.txt") -> list[GoldenCase]:
    cases, cur = [], None
    with open(os.path.join(GOLDEN_DIR, filename), encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = {"name": line[1:-1]}
                cases.append(cur)
                continue
            key, _, val = line.partition("=")
            cur[key.strip()] = val.strip()
    out = []
    for c in cases:
        tokens = np.array(_ints(c["tokens"]), dtype=np.int32)
        offsets = np.array(_ints(c.get("offsets", f"0 {tokens.size}")), dtype=np.int64)
        B, K = offsets.size - 1, int(c["K"])

        def per_request(key: str) -> list[str]:
            parts = [p.strip() for p in c[key].split("|")]
            assert len(parts) == B, (c["name"], key)
            return parts

        draft = np.array([_ints(p) for p in per_request("expect_draft")],
                         dtype=np.int32).reshape(B, K)
        out.append(GoldenCase(
            c["name"], tokens, offsets, int(c["min_m"]), int(c["max_m"]), K,
            np.array([int(p) for p in per_request("expect_m")], dtype=np.int32),
            np.array([int(p) for p in per_request("expect_pos")], dtype=np.int32),
            np.array([int(p) for p in per_request("expect_len")], dtype=np.int32),
            draft))
    return out
