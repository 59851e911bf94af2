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


def support_order(rows: np.ndarray, n: int, m: int) -> Tuple[np.ndarray, np.ndarray]:
    """The table with its attributes in ascending support order, ties by attribute index: the
    library's default processing order. Returns (permuted packed rows, inv) where inv[r] is the
    attribute at position r. The output set of an enumeration does not depend on the order; the
    number of candidates it evaluates does."""
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    wm = (m + 31) // 32
    bits = np.unpackbits(rows.view(np.uint8), bitorder="little").reshape(n, wm * 32)[:, :m]
    inv = np.argsort(bits.sum(axis=0), kind="stable")
    pad = np.zeros((n, wm * 32), dtype=np.uint8)
    pad[:, :m] = bits[:, inv]
    return np.packbits(pad, axis=1, bitorder="little").view(np.uint32).reshape(n, wm).copy(), inv


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


_M1, _M2 = np.uint64(0xBF58476D1CE4E5B9), np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def multiset_digest(intents: np.ndarray, chunk: int = 1 << 22):
    """Order-independent digest of a set of intents: (sum, xor) mod 2^64 of one hash per row.

    The hash folds the row's 32-bit words in order through the splitmix64 finaliser and then the
    word count (the same definition as the oracle's digest mode).
    """
    rows = np.ascontiguousarray(intents, dtype=np.uint32)
    k, w = rows.shape
    hsum, hxor = np.uint64(0), np.uint64(0)
    with np.errstate(over="ignore"):
        for lo in range(0, k, chunk):
            part = rows[lo:lo + chunk].astype(np.uint64)
            h = np.full(part.shape[0], 0x9E3779B97F4A7C15, dtype=np.uint64)
            for i in range(w):
                h = _mix64(h ^ part[:, i])
            h = _mix64(h + np.uint64(w))
            hsum = np.uint64(hsum + np.sum(h, dtype=np.uint64))
            hxor = np.uint64(hxor ^ np.bitwise_xor.reduce(h))
    return int(hsum), int(hxor)
