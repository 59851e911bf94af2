"""Seeded synthetic formal contexts (binary object x attribute tables).

This module only draws and packs 0/1 tables; it holds none of the concept
enumeration arithmetic. Tests, the benchmark and the oracle-side checks all
take their inputs from here, so both the CUDA library and the CPU oracle see
exactly the same bytes.

Packing convention (Parallel FCBO page, section 3.1 column-bitmap listing;
FCbO-to-CUDA page, section 4.3 canonical mask): attribute ``a`` of an object
is bit ``a & 31`` of 32-bit word ``a >> 5`` of that object's row, least
significant bit first. Padding bits past ``M`` are zero.

The five named workloads stand in for the pages' anonymous datasets
(FCbO-to-CUDA page, section 5.1: an e-commerce context of 68,000 x 412 and a
software-configuration context of 1,920 x 96), which are not available.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Dict, Tuple

import numpy as np


def words32(n_bits: int) -> int:
    """Number of 32-bit words that hold ``n_bits`` bits (ceil, never floor)."""
    return (int(n_bits) + 31) // 32


def pack_rows(cells: np.ndarray) -> np.ndarray:
    """Pack a boolean ``(N, M)`` table into ``(N, ceil(M/32))`` uint32 rows, LSB-first."""
    cells = np.ascontiguousarray(cells, dtype=bool)
    n, m = cells.shape
    wm = words32(m)
    padded = np.zeros((n, wm * 32), dtype=bool)
    padded[:, :m] = cells
    packed = np.packbits(padded, axis=1, bitorder="little")  # (n, wm*4) bytes
    return np.ascontiguousarray(packed).view("<u4").astype(np.uint32).reshape(n, wm)


def unpack_rows(rows: np.ndarray, m: int) -> np.ndarray:
    """Inverse of :func:`pack_rows`: ``(N, W)`` uint32 rows -> boolean ``(N, m)``."""
    rows = np.ascontiguousarray(rows, dtype="<u4")
    n = rows.shape[0]
    as_bytes = rows.view(np.uint8).reshape(n, -1)
    bits = np.unpackbits(as_bytes, axis=1, bitorder="little")
    return bits[:, :m].astype(bool)


def bernoulli_cells(n: int, m: int, p_col: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    """One ``rng.random((n, m))`` draw (row-major), compared with a per-column probability."""
    u = rng.random((n, m))
    return u < np.asarray(p_col, dtype=np.float64)[None, :]


def zipf_profile(m: int, s: float, mean: float) -> np.ndarray:
    """Per-attribute densities ``min(1, c * (k+1)^-s)`` with ``c`` bisected to the target mean."""
    base = (np.arange(m, dtype=np.float64) + 1.0) ** (-s)
    lo, hi = 0.0, 1.0 / base.min()
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if np.minimum(1.0, mid * base).mean() < mean:
            lo = mid
        else:
            hi = mid
    return np.minimum(1.0, 0.5 * (lo + hi) * base)


@dataclass(frozen=True)
class Workload:
    name: str
    n_objects: int
    n_attrs: int
    seed: int
    description: str
    make_cells: Callable[[], np.ndarray]

    def cells(self) -> np.ndarray:
        return self.make_cells()

    def rows(self) -> np.ndarray:
        return pack_rows(self.make_cells())


def _tiny() -> np.ndarray:
    rng = np.random.default_rng(0)
    return bernoulli_cells(64, 16, np.full(16, 0.3), rng)


def _sparse() -> np.ndarray:
    rng = np.random.default_rng(1)
    return bernoulli_cells(2000, 64, np.full(64, 0.15), rng)


def _skewed() -> np.ndarray:
    rng = np.random.default_rng(2)
    p = np.empty(128)
    p[0:8] = 0.9
    p[8:32] = 0.3
    p[32:128] = 0.03
    return bernoulli_cells(10000, 128, p, rng)


def _zipf() -> np.ndarray:
    rng = np.random.default_rng(3)
    return bernoulli_cells(50000, 400, zipf_profile(400, 1.1, 0.02), rng)


def planted_cells(n: int, m: int, p: float, blocks: int, objects: Tuple[int, int], attrs: Tuple[int, int],
                  rng: np.random.Generator) -> np.ndarray:
    """Bernoulli(p) background, then `blocks` all-ones blocks set in order: for each, a number of
    objects drawn from [objects[0], objects[1]] and of attributes from [attrs[0], attrs[1]], then
    that many distinct objects and attributes (blocks may overlap)."""
    cells = bernoulli_cells(n, m, np.full(m, p), rng)
    for _ in range(blocks):
        no = int(rng.integers(objects[0], objects[1] + 1))
        na = int(rng.integers(attrs[0], attrs[1] + 1))
        objs = rng.choice(n, no, replace=False)
        cols = rng.choice(m, na, replace=False)
        cells[np.ix_(objs, cols)] = True
    return cells


def _biclusters() -> np.ndarray:
    return planted_cells(100000, 256, 0.01, 40, (500, 5000), (6, 20), np.random.default_rng(4))


def _biclusters_50k() -> np.ndarray:
    # the same recipe at half the objects and blocks: a case small enough for multi-pass profiling
    return planted_cells(50000, 256, 0.01, 20, (500, 5000), (6, 20), np.random.default_rng(5))


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny", 64, 16, 0, "64x16 Bernoulli(0.3)", _tiny),
        Workload("sparse", 2000, 64, 1, "2,000x64 Bernoulli(0.15)", _sparse),
        Workload("skewed", 10000, 128, 2,
                 "10,000x128; attrs 0-7 p=0.9, 8-31 p=0.3, 32-127 p=0.03", _skewed),
        Workload("zipf", 50000, 400, 3,
                 "50,000x400; per-attribute Zipf(s=1.1) densities, mean 0.02", _zipf),
        Workload("biclusters", 100000, 256, 4,
                 "100,000x256; Bernoulli(0.01) background + 40 planted blocks", _biclusters),
        Workload("biclusters_50k", 50000, 256, 5,
                 "50,000x256; Bernoulli(0.01) background + 20 planted blocks", _biclusters_50k),
    ]
}


def random_context(n: int, m: int, density: float, seed: int) -> np.ndarray:
    """Packed rows of an i.i.d. Bernoulli(density) context (test helper)."""
    rng = np.random.default_rng(seed)
    return pack_rows(bernoulli_cells(n, m, np.full(m, density), rng))


def planted_context(n: int, m: int, p: float, blocks: int, objects: Tuple[int, int], attrs: Tuple[int, int],
                    seed: int) -> np.ndarray:
    """Packed rows of a small planted-block context (test helper; the recipe of the planted-bicluster
    workload at other sizes)."""
    return pack_rows(planted_cells(n, m, p, blocks, objects, attrs, np.random.default_rng(seed)))


def contranominal(n: int) -> np.ndarray:
    """Object i has every attribute except i (n x n)."""
    return pack_rows(~np.eye(n, dtype=bool))


def identity(n: int) -> np.ndarray:
    """Object i has only attribute i (n x n)."""
    return pack_rows(np.eye(n, dtype=bool))
