"""Concept-lattice oracle: extents of intents and the cover relation — TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may use this module. The
CUDA library never calls it and shares no code with it.

Definitions (FCbO-to-CUDA article, sections 1.1 and 4.4; Parallel FCBO article, sections 1.1 and
3.4): concepts are ordered by extent inclusion, (A1, B1) <= (A2, B2) iff A1 is a subset of A2, which
holds iff B1 contains B2. Concept j is a lower cover of concept i when intent_i is a proper subset of
intent_j and no intent lies strictly between them. The articles draw the lattice from these edges;
the search tree's parent-child links are not them.

  * :func:`cover_edges`       every cover edge of a whole intent set, written as the definition with a
                              Boolean matrix product (K <= a few thousand);
  * :func:`lower_covers_of`   the lower covers of one concept against a whole intent set (any K),
                              for sampled checks of large sets.
"""
from __future__ import annotations

import numpy as np


def _bits(intents: np.ndarray, n_attrs: int) -> np.ndarray:
    """Intents as a (K, M) boolean matrix (attribute a = bit a & 31 of word a >> 5)."""
    x = np.ascontiguousarray(intents, dtype=np.uint32)
    cells = np.unpackbits(x.view(np.uint8), axis=1, bitorder="little")
    return cells[:, :n_attrs].astype(bool)


def cover_edges(intents: np.ndarray, n_attrs: int) -> np.ndarray:
    """All cover edges (i, j), j a lower cover of i, as a sorted (E, 2) int64 array of row indices.

    proper[i, j] = intent_i is a proper subset of intent_j (attribute-set inclusion, written as "no
    attribute of i outside j" and "j has more attributes"); j covers i from below when proper[i, j]
    holds and no k has proper[i, k] and proper[k, j], the second condition taken from the Boolean
    product of proper with itself.
    """
    cells = _bits(intents, n_attrs)
    k = cells.shape[0]
    if k == 0:
        return np.zeros((0, 2), dtype=np.int64)
    c = cells.astype(np.float32)
    size = cells.sum(axis=1)
    # attributes of i missing from j: |B_i| - |B_i & B_j|
    outside = size[:, None] - (c @ c.T)
    proper = (outside == 0) & (size[None, :] > size[:, None])
    p = proper.astype(np.float32)
    between = (p @ p) > 0
    cover = proper & ~between
    i, j = np.nonzero(cover)
    return np.stack([i, j], axis=1).astype(np.int64)


def lower_covers_of(intents: np.ndarray, n_attrs: int, i: int) -> np.ndarray:
    """Row indices j (ascending) of the lower covers of concept i within the set ``intents``.

    The proper supersets of intent_i are found by a scan of the whole set; the lower covers are the
    minimal ones under inclusion. They are taken out in order of size: the smallest superset left is
    minimal (a superset inside it would be smaller, and would either still be left or have gone with
    a minimal one that is then inside it too), and every superset containing it is dropped with it.
    """
    x = np.ascontiguousarray(intents, dtype=np.uint32)
    b = x[i]
    sup = np.nonzero(np.all((x & b[None, :]) == b[None, :], axis=1))[0]
    sup = sup[sup != i]
    size = _bits(x[sup], n_attrs).sum(axis=1) if sup.size else np.zeros(0, dtype=np.int64)
    left = sup[np.argsort(size, kind="stable")]
    covers = []
    while left.size:
        c = left[0]
        covers.append(c)
        inside = np.all((x[left] & x[c][None, :]) == x[c][None, :], axis=1)
        left = left[~inside]
    return np.sort(np.asarray(covers, dtype=np.int64))
