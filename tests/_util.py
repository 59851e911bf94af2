"""Comparison helpers for the tests (no enumeration arithmetic here)."""
from __future__ import annotations

import os
from typing import List, Tuple

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def sort_rows(rows: np.ndarray) -> np.ndarray:
    """Rows of uint32 words sorted ascending as big integers (last word most significant)."""
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    if rows.ndim != 2 or rows.shape[0] == 0:
        return rows
    return rows[np.lexsort(rows.T)]


def same_set(a: np.ndarray, b: np.ndarray) -> bool:
    a, b = sort_rows(a), sort_rows(b)
    return a.shape == b.shape and bool(np.array_equal(a, b))


def has_duplicates(rows: np.ndarray) -> bool:
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    return np.unique(rows, axis=0).shape[0] != rows.shape[0]


def attrs_to_row(attrs, m: int) -> np.ndarray:
    row = np.zeros((m + 31) // 32, dtype=np.uint32)
    for a in attrs:
        row[a >> 5] |= np.uint32(1 << (a & 31))
    return row


def load_golden(name: str) -> Tuple[int, int, np.ndarray, np.ndarray]:
    """(N, M, packed rows, expected intents) of a hand-derived fixture."""
    n = m = None
    rows: List[List[int]] = []
    intents: List[List[int]] = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "n":
                n = int(vals[0])
            elif key == "m":
                m = int(vals[0])
            elif key == "row":
                rows.append([int(v) for v in vals])
            elif key == "intent":
                intents.append([int(v) for v in vals])
    assert n == len(rows)
    packed = np.stack([attrs_to_row(r, m) for r in rows])
    expected = np.stack([attrs_to_row(i, m) for i in intents])
    return n, m, packed, expected


def golden_names() -> List[str]:
    return sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt"))
