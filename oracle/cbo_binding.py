"""ctypes binding of the C Close-by-One oracle (test infrastructure only)."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cbo.c")
_LIB_PATH = os.path.join(_HERE, "libcbo_oracle.so")
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def oracle_library_path() -> str:
    return _LIB_PATH


def build_oracle(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``cbo.c`` with gcc into a shared library (portable flags only)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed). ``path`` loads another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build_oracle()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    u32pp = ctypes.POINTER(ctypes.POINTER(ctypes.c_uint32))
    lib.oracle_cbo.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int, ctypes.c_int,
        u32pp, u32pp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
        ctypes.c_void_p,
    ]
    lib.oracle_cbo.restype = ctypes.c_int
    lib.oracle_cbo_limited.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
        u32pp, u32pp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
        ctypes.c_void_p,
    ]
    lib.oracle_cbo_limited.restype = ctypes.c_int
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.oracle_cbo_digest.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                                      u64p, u64p, ctypes.c_void_p, u64p, u64p]
    lib.oracle_cbo_digest.restype = ctypes.c_int
    lib.oracle_cbo_digest_relabel.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                                              ctypes.c_void_p, u64p, u64p, ctypes.c_void_p, u64p, u64p]
    lib.oracle_cbo_digest_relabel.restype = ctypes.c_int
    lib.oracle_free.argtypes = [ctypes.c_void_p]
    lib.oracle_free.restype = None
    return lib


def cbo(rows: np.ndarray, n_objects: int, n_attrs: int, threads: int = 1,
        want_extents: bool = False, lib: Optional[ctypes.CDLL] = None, limit: int = 0) -> dict:
    """Run the recursive CbO oracle.

    ``rows``: ``(N, ceil(M/32))`` uint32 packed rows. Returns a dict with
    ``intents`` (K x ceil(M/32) uint32, output order of the search), ``extents``
    (K x ceil(N/32) uint32 or None), ``closures`` (candidates evaluated),
    ``depth_counts`` (concepts per search depth, length M+2). ``limit`` > 0
    stops each thread after that many intents (a bounded timing sample).
    """
    lib = lib or load()
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    wm = (n_attrs + 31) // 32
    wn = (n_objects + 31) // 32
    if rows.shape != (n_objects, wm):
        raise ValueError(f"rows shape {rows.shape} != {(n_objects, wm)}")
    p_int = ctypes.POINTER(ctypes.c_uint32)()
    p_ext = ctypes.POINTER(ctypes.c_uint32)()
    count = ctypes.c_uint64(0)
    closures = ctypes.c_uint64(0)
    depth = np.zeros(n_attrs + 2, dtype=np.uint64)
    if limit:
        rc = lib.oracle_cbo_limited(rows.ctypes.data, n_objects, n_attrs, int(threads), int(want_extents),
                                    int(limit), ctypes.byref(p_int), ctypes.byref(p_ext),
                                    ctypes.byref(count), ctypes.byref(closures), depth.ctypes.data)
    else:
        rc = lib.oracle_cbo(rows.ctypes.data, n_objects, n_attrs, int(threads), int(want_extents),
                            ctypes.byref(p_int), ctypes.byref(p_ext), ctypes.byref(count),
                            ctypes.byref(closures), depth.ctypes.data)
    if rc != 0:
        raise RuntimeError("oracle_cbo failed (bad arguments or out of memory)")
    k = int(count.value)
    try:
        intents = np.ctypeslib.as_array(p_int, shape=(max(k, 1) * wm,))[: k * wm].copy().reshape(k, wm)
        extents = None
        if want_extents:
            extents = np.ctypeslib.as_array(p_ext, shape=(max(k, 1) * wn,))[: k * wn].copy().reshape(k, wn)
    finally:
        lib.oracle_free(ctypes.cast(p_int, ctypes.c_void_p))
        if want_extents:
            lib.oracle_free(ctypes.cast(p_ext, ctypes.c_void_p))
    return {"intents": intents, "extents": extents, "closures": int(closures.value),
            "depth_counts": depth}


def cbo_digest(rows: np.ndarray, n_objects: int, n_attrs: int, threads: int = 1,
               lib: Optional[ctypes.CDLL] = None, label: Optional[np.ndarray] = None) -> dict:
    """The same search keeping no intents: their number, the closures, the depth counts and an
    order-independent digest of the intent set (sum and xor mod 2^64 of one hash per intent).

    ``label`` (optional, a permutation of 0..M-1): the table's attribute at position r is attribute
    ``label[r]`` of the original table; the digest is then taken over the intents renumbered back to
    the original attributes (the closures stay those of the search in the given order)."""
    lib = lib or load()
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    if rows.shape != (n_objects, (n_attrs + 31) // 32):
        raise ValueError("rows shape does not match (N, ceil(M/32))")
    count, closures = ctypes.c_uint64(0), ctypes.c_uint64(0)
    hsum, hxor = ctypes.c_uint64(0), ctypes.c_uint64(0)
    depth = np.zeros(n_attrs + 2, dtype=np.uint64)
    if label is not None:
        lab = np.ascontiguousarray(label, dtype=np.int32)
        if lab.shape != (n_attrs,):
            raise ValueError("label must hold one attribute number per column")
        rc = lib.oracle_cbo_digest_relabel(rows.ctypes.data, n_objects, n_attrs, int(threads), lab.ctypes.data,
                                           ctypes.byref(count), ctypes.byref(closures), depth.ctypes.data,
                                           ctypes.byref(hsum), ctypes.byref(hxor))
    else:
        rc = lib.oracle_cbo_digest(rows.ctypes.data, n_objects, n_attrs, int(threads), ctypes.byref(count),
                                   ctypes.byref(closures), depth.ctypes.data, ctypes.byref(hsum),
                                   ctypes.byref(hxor))
    if rc != 0:
        raise RuntimeError("oracle_cbo_digest failed")
    return {"count": int(count.value), "closures": int(closures.value), "depth_counts": depth,
            "hsum": int(hsum.value), "hxor": int(hxor.value)}
