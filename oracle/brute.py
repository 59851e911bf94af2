"""Brute-force closure of every attribute subset, and the two derivation operators.

Test infrastructure only. These restate the definitions of the FCbO-to-CUDA
page, section 1.1 (Y' = objects having every attribute of Y; X' = attributes
shared by every object of X; a concept is a pair with X' = Y and Y' = X) and
the Parallel FCBO page, section 1.1 (B is closed iff B'' = B), with numpy on
packed bitmaps. No search order, pruning or canonical test is involved, so
they pin the recursive oracle from outside.
"""
from __future__ import annotations

import numpy as np


def _full_intent(n_attrs: int) -> np.ndarray:
    wm = (n_attrs + 31) // 32
    out = np.zeros(wm, dtype=np.uint32)
    for a in range(n_attrs):
        out[a >> 5] |= np.uint32(1 << (a & 31))
    return out


def derive_extent(rows: np.ndarray, intent: np.ndarray) -> np.ndarray:
    """Y': boolean mask of the objects whose row contains every attribute of ``intent``."""
    rows = np.asarray(rows, dtype=np.uint32)
    intent = np.asarray(intent, dtype=np.uint32)
    return np.all((rows & intent[None, :]) == intent[None, :], axis=1)


def derive_intent(rows: np.ndarray, extent_mask: np.ndarray, n_attrs: int) -> np.ndarray:
    """X': AND of the rows of the objects in ``extent_mask``; the empty set gives all attributes."""
    rows = np.asarray(rows, dtype=np.uint32)
    sel = rows[np.asarray(extent_mask, dtype=bool)]
    full = _full_intent(n_attrs)
    if sel.shape[0] == 0:
        return full
    return np.bitwise_and.reduce(sel, axis=0) & full


def brute_force(rows: np.ndarray, n_objects: int, n_attrs: int) -> np.ndarray:
    """All distinct closures S'' over every subset S of the attributes (M <= 20).

    Returns a ``(K, ceil(M/32))`` uint32 array, rows sorted ascending as integers.
    """
    if n_attrs > 20:
        raise ValueError("brute force is for M <= 20")
    rows = np.asarray(rows, dtype=np.uint32).reshape(n_objects, -1)
    r = rows[:, 0].astype(np.int64)                 # M <= 20 fits in word 0
    full = (1 << n_attrs) - 1
    seen = set()
    subsets = np.arange(1 << n_attrs, dtype=np.int64)
    step = 4096
    for lo in range(0, subsets.size, step):
        s = subsets[lo:lo + step]
        # has[i, o]: object o has every attribute of subset i   (S')
        has = (r[None, :] & s[:, None]) == s[:, None]
        # S'' = AND over those objects' rows, all attributes when none
        vals = np.where(has, r[None, :], full)
        closed = np.bitwise_and.reduce(vals, axis=1) & full
        seen.update(int(v) for v in np.unique(closed))
    out = np.array(sorted(seen), dtype=np.uint32).reshape(-1, 1)
    return out


def brute_force_by_objects(rows: np.ndarray, n_objects: int, n_attrs: int) -> np.ndarray:
    """All intents as derivations Y' of every object subset Y (N <= 16, any M).

    Every intent is B = B'' = (B')', the derivation of an object set, and every
    derivation Y' of an object set is closed (Y' = Y'''), so the intents are
    exactly {Y' : Y subset of the objects}; Y = empty gives all M attributes.
    Returns ``(K, ceil(M/32))`` uint32 rows, sorted ascending as integers
    (last word most significant).
    """
    if n_objects > 16:
        raise ValueError("object brute force is for N <= 16")
    rows = np.asarray(rows, dtype=np.uint32).reshape(n_objects, -1)
    full = _full_intent(n_attrs)
    # derivations of all subsets of the first k objects, doubled one object at a time
    acc = full[None, :].copy()
    for o in range(n_objects):
        acc = np.concatenate([acc, acc & rows[o][None, :]], axis=0)
    uniq = np.unique(acc, axis=0)
    order = np.lexsort(uniq.T)          # last word is the most significant key
    return np.ascontiguousarray(uniq[order])
