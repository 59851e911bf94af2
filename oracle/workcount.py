"""ctypes binding of the work-counting pass in ``workcount.c`` (test and measurement infrastructure).

``workcount(rows, n, m, mid_max=T)`` returns, per tier, the algorithmic work of enumerating the
context in 32-bit words: the units and the per-unit counts that the roofline uses (see the header
of ``workcount.c``). Tier ``"list"`` holds the parents with at most 64 objects, tier ``"mid"`` those
with at most T objects (none when T <= 64), tier ``"bitmap"`` the larger ones.

``coverwork(rows, n, m, intents)`` returns the work of the lower-cover search over an intent set
(see the header of ``coverwork.c``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "workcount.c")
_SRCS = (_SRC, os.path.join(_HERE, "coverwork.c"))
_LIB_PATH = os.path.join(_HERE, "libworkcount.so")
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

FIELDS = ("parents", "closures", "children", "isect_words", "closure_words", "canon_words", "hbm_words",
          "hbm_lean_words", "l2_lean_words")
TIERS = ("list", "mid", "bitmap")


def build(force: bool = False) -> str:
    """Compile ``workcount.c`` and ``coverwork.c`` with gcc into a shared library (portable flags only)."""
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src) for src in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", *_SRCS, "-o", tmp], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.workcount.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                                      ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint64)]
            lib.workcount.restype = ctypes.c_int
            lib.coverwork.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]
            lib.coverwork.restype = ctypes.c_int
            _lib = lib
    return _lib


def workcount(rows: np.ndarray, n_objects: int, n_attrs: int, threads: int = 1,
              mid_max: int = 0, list_max: int = 0) -> Dict[str, Dict[str, int]]:
    """Per-tier work counts of enumerating ``rows`` (``N x ceil(M/32)`` uint32, LSB-first). The lean
    model's fields depend on ``list_max`` (largest extent kept as an id list; 0: none)."""
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    out = (ctypes.c_uint64 * 27)()
    st = _load().workcount(rows.ctypes.data, int(n_objects), int(n_attrs), int(threads), int(mid_max),
                           int(list_max), out)
    if st != 0:
        raise RuntimeError("workcount failed")
    return {t: {f: int(out[9 * i + k]) for k, f in enumerate(FIELDS)} for i, t in enumerate(TIERS)}


def derived(counts: Dict[str, int]) -> Dict[str, int]:
    """Words read from L2 (intersection and closure), word operations, and HBM words of one tier."""
    l2 = counts["isect_words"] + counts["closure_words"]
    return {"l2_words": l2, "ops": l2 + counts["canon_words"], "hbm_words": counts["hbm_words"]}


COVER_FIELDS = ("concepts", "extent_words", "isect_words", "closure_words")


def coverwork(rows: np.ndarray, n_objects: int, n_attrs: int, intents: np.ndarray, threads: int = 1) -> Dict[str, int]:
    """Work of the lower-cover search over ``intents`` (``K x ceil(M/32)`` uint32) of the context
    ``rows``: per concept its extent once, the intersections A & column k for k outside B over the
    non-zero words of A, and the closure of each non-empty one as the AND of its objects' rows."""
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    intents = np.ascontiguousarray(intents, dtype=np.uint32)
    wm = (n_attrs + 31) // 32
    if intents.ndim != 2 or intents.shape[1] != wm:
        raise ValueError("intents must be K x ceil(M/32) words")
    out = (ctypes.c_uint64 * 4)()
    st = _load().coverwork(rows.ctypes.data, int(n_objects), int(n_attrs),
                           intents.ctypes.data if intents.shape[0] else None, int(intents.shape[0]), int(threads), out)
    if st != 0:
        raise RuntimeError("coverwork failed")
    return {f: int(out[i]) for i, f in enumerate(COVER_FIELDS)}
