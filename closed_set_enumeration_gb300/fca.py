"""Thin ctypes binding of libfca (the C ABI in include/fca.h).

Argument marshalling only: every step of the enumeration runs in the CUDA
library. PyTorch is used for device memory and streams. There is no CPU
fallback: if libfca.so is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfca.so")

FCA_OK, FCA_ERR_INVALID, FCA_ERR_OOM, FCA_ERR_CAPACITY, FCA_ERR_CUDA = range(5)

# Every entry point declared in include/fca.h.
EXPORTS = (
    "fca_context_create", "fca_context_load", "fca_enumerate", "fca_enumerate_host", "fca_set_option",
    "fca_get_stats", "fca_context_dims", "fca_context_copy", "fca_last_error", "fca_free", "fca_status_string",
    "fca_enumerate_small_noalloc", "fca_extents", "fca_cover_edges",
)


FCA_OPT_COUNT_WORK, FCA_OPT_LEVEL_BYTES, FCA_OPT_QUEUE_ENTRIES, FCA_OPT_POOL_LIMIT_BYTES = 1, 2, 3, 4
FCA_OPT_ATTR_ORDER = 5
FCA_OPT_WAIT_LIMIT_NS = 6


class FcaStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_uint64) for name in (
        "concepts", "closures", "large_parents", "small_roots", "launches", "levels",
        "max_frontier", "frontier_bytes", "expand_launches", "subtree_launches",
        "subtree_word_ops", "expand_bytes", "retries", "spill_rounds")] + [("expand_ms", ctypes.c_double),
                                                ("subtree_ms", ctypes.c_double),
                                                ("lattice_ms", ctypes.c_double),
                                                ("mid_launches", ctypes.c_uint64),
                                                ("mid_ms", ctypes.c_double),
                                                ("list_max", ctypes.c_uint64),
                                                ("mid_max", ctypes.c_uint64)]

    def as_dict(self) -> dict:
        return {name: (float(getattr(self, name)) if ty is ctypes.c_double else int(getattr(self, name)))
                for name, ty in self._fields_}


class FcaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfca.so; raise if it was not built (no fallback of any kind)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libfca.so not found at {path}; build it with "
                              "closed_set_enumeration_gb300.build.build()")
        lib = ctypes.CDLL(path)
        vp, u64, i64, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32
        lib.fca_context_create.argtypes = [vp, i64, i32, ctypes.POINTER(vp)]
        lib.fca_context_load.argtypes = [vp, vp, vp]
        lib.fca_enumerate.argtypes = [vp, vp, u64, ctypes.POINTER(u64), vp]
        lib.fca_enumerate_host.argtypes = [vp, vp, u64, ctypes.POINTER(u64), vp]
        lib.fca_set_option.argtypes = [vp, ctypes.c_int, i64]
        lib.fca_extents.argtypes = [vp, vp, u64, vp, vp]
        lib.fca_cover_edges.argtypes = [vp, vp, u64, vp, u64, ctypes.POINTER(u64), vp]
        lib.fca_enumerate_small_noalloc.argtypes = [vp, i64, i32, vp, u64, ctypes.POINTER(u64), vp]
        lib.fca_enumerate_small_noalloc.restype = ctypes.c_int
        lib.fca_get_stats.argtypes = [vp, ctypes.POINTER(FcaStats)]
        lib.fca_context_dims.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i32)]
        lib.fca_context_copy.argtypes = [vp, ctypes.c_int, vp, u64]
        lib.fca_last_error.argtypes = [vp]
        lib.fca_last_error.restype = ctypes.c_char_p
        lib.fca_free.argtypes = [vp]
        lib.fca_free.restype = None
        lib.fca_status_string.argtypes = [ctypes.c_int]
        lib.fca_status_string.restype = ctypes.c_char_p
        for name in ("fca_context_create", "fca_context_load", "fca_enumerate", "fca_enumerate_host", "fca_set_option", "fca_get_stats",
                     "fca_context_dims", "fca_context_copy", "fca_extents", "fca_cover_edges"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().fca_status_string(int(status)).decode()


def words(n_bits: int) -> int:
    return (int(n_bits) + 31) // 32


def _ptr(x) -> int:
    """Raw address of a numpy array or torch tensor (contiguous)."""
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return x.ctypes.data
    import torch
    if isinstance(x, torch.Tensor):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr()
    raise TypeError(f"unsupported buffer type {type(x)}")


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Context:
    """A formal context resident on the current CUDA device.

    ``rows``: ``(N, ceil(M/32))`` uint32 row bitmaps (numpy array on the host,
    or a torch tensor on the host or the device, any 32-bit dtype).
    """

    def __init__(self, rows, n_objects: int, n_attrs: int):
        self._lib = load_library()
        self.n_objects = int(n_objects)
        self.n_attrs = int(n_attrs)
        self.wm = words(n_attrs)
        self._h = ctypes.c_void_p()
        if isinstance(rows, np.ndarray):
            rows = np.ascontiguousarray(rows, dtype=np.uint32)
        if tuple(rows.shape) != (self.n_objects, self.wm):
            raise ValueError(f"rows shape {tuple(rows.shape)} != {(self.n_objects, self.wm)}")
        self._keep = rows
        st = self._lib.fca_context_create(ctypes.c_void_p(_ptr(rows)), self.n_objects, self.n_attrs,
                                          ctypes.byref(self._h))
        self._keep = None
        if st != FCA_OK:
            raise FcaError(st, f"fca_context_create: {status_string(st)}")

    # --------------------------------------------------------------- lifetime
    def close(self) -> None:
        if self._h:
            self._lib.fca_free(self._h)
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st: int, what: str, allow_capacity: bool = False) -> None:
        if st == FCA_OK or (allow_capacity and st == FCA_ERR_CAPACITY):
            return
        msg = self._lib.fca_last_error(self._h)
        raise FcaError(st, f"{what}: {status_string(st)}: {msg.decode() if msg else ''}")

    # --------------------------------------------------------------- calls
    def load(self, rows, stream=None) -> None:
        """Replace the table with new rows of the same shape (host array or host/device tensor)."""
        if isinstance(rows, np.ndarray):
            rows = np.ascontiguousarray(rows, dtype=np.uint32)
        if tuple(rows.shape) != (self.n_objects, self.wm):
            raise ValueError(f"rows shape {tuple(rows.shape)} != {(self.n_objects, self.wm)}")
        st = self._lib.fca_context_load(self._h, ctypes.c_void_p(_ptr(rows)),
                                        ctypes.c_void_p(_stream_handle(stream)))
        self._check(st, "fca_context_load")

    def enumerate_into(self, out, capacity: Optional[int] = None, stream=None) -> Tuple[int, int]:
        """Enumerate into a caller-owned device buffer ``out`` (``capacity x W_M`` words).

        Returns ``(status, count)``; status is FCA_OK or FCA_ERR_CAPACITY.
        """
        cap = int(out.shape[0]) if capacity is None else int(capacity)
        count = ctypes.c_uint64(0)
        ptr = _ptr(out) if cap > 0 else 0
        st = self._lib.fca_enumerate(self._h, ctypes.c_void_p(ptr), cap, ctypes.byref(count),
                                     ctypes.c_void_p(_stream_handle(stream)))
        self._check(st, "fca_enumerate", allow_capacity=True)
        return st, int(count.value)

    def enumerate(self, capacity: Optional[int] = None, stream=None):
        """All intents as a device tensor ``(K, W_M)`` (int32 holding the uint32 words).

        Retries once with the exact size when ``capacity`` is too small.
        """
        import torch
        cap = int(capacity) if capacity is not None else 1 << 16
        while True:
            out = torch.empty((max(cap, 1), self.wm), dtype=torch.int32, device="cuda")
            st, count = self.enumerate_into(out, cap, stream)
            if st == FCA_OK:
                return out[:count]
            cap = count

    def enumerate_host(self, out_host: np.ndarray, stream=None) -> Tuple[int, int]:
        """Enumerate into a host array ``out_host`` (``capacity x W_M`` uint32)."""
        count = ctypes.c_uint64(0)
        cap = int(out_host.shape[0])
        st = self._lib.fca_enumerate_host(self._h, ctypes.c_void_p(_ptr(out_host) if cap else 0), cap,
                                          ctypes.byref(count), ctypes.c_void_p(_stream_handle(stream)))
        self._check(st, "fca_enumerate_host", allow_capacity=True)
        return st, int(count.value)

    def extents(self, intents, stream=None):
        """Extent of each row of the device tensor ``intents`` (``K x W_M`` 32-bit words, attribute
        order) as a device tensor ``(K, W_N)`` (int32 holding the uint32 words, objects LSB first)."""
        import torch
        out = torch.empty((int(intents.shape[0]), words(self.n_objects)), dtype=torch.int32, device=intents.device)
        self.extents_into(intents, out, stream)
        return out

    def extents_into(self, intents, out, stream=None) -> None:
        """Extents of the rows of ``intents`` into the caller's device buffer ``out`` (``K x W_N`` words);
        enqueued on ``stream`` without waiting."""
        k = int(intents.shape[0])
        if k:
            st = self._lib.fca_extents(self._h, ctypes.c_void_p(_ptr(intents)), k, ctypes.c_void_p(_ptr(out)),
                                       ctypes.c_void_p(_stream_handle(stream)))
            self._check(st, "fca_extents")

    def enumerate_concepts(self, capacity: Optional[int] = None, stream=None):
        """All concepts as two device tensors: intents ``(K, W_M)`` and their extents ``(K, W_N)``."""
        intents = self.enumerate(capacity, stream)
        return intents, self.extents(intents, stream)

    def cover_edges_into(self, intents, edges, capacity: Optional[int] = None, stream=None) -> Tuple[int, int]:
        """Cover edges of the complete intent set ``intents`` into the caller's device buffer ``edges``
        (``capacity x 2`` 32-bit words). Returns ``(status, edge count)``."""
        cap = int(edges.shape[0]) if capacity is None else int(capacity)
        n = ctypes.c_uint64(0)
        st = self._lib.fca_cover_edges(self._h, ctypes.c_void_p(_ptr(intents)), int(intents.shape[0]),
                                       ctypes.c_void_p(_ptr(edges) if cap else 0), cap, ctypes.byref(n),
                                       ctypes.c_void_p(_stream_handle(stream)))
        self._check(st, "fca_cover_edges", allow_capacity=True)
        return st, int(n.value)

    def cover_edges(self, intents, capacity: Optional[int] = None, stream=None):
        """Cover edges (upper row, lower row) of the complete intent set ``intents`` as a device tensor
        ``(E, 2)`` (int32 holding row indices). Retries once with the exact size when needed."""
        import torch
        cap = int(capacity) if capacity is not None else max(64, 4 * int(intents.shape[0]))
        while True:
            out = torch.empty((max(cap, 1), 2), dtype=torch.int32, device=intents.device)
            st, n = self.cover_edges_into(intents, out, cap, stream)
            if st == FCA_OK:
                return out[:n]
            cap = n

    def set_option(self, option: int, value: int) -> None:
        self._check(self._lib.fca_set_option(self._h, int(option), int(value)), "fca_set_option")

    def stats(self) -> dict:
        s = FcaStats()
        self._check(self._lib.fca_get_stats(self._h, ctypes.byref(s)), "fca_get_stats")
        return s.as_dict()

    def dims(self) -> Tuple[int, int]:
        n = ctypes.c_int64()
        m = ctypes.c_int32()
        self._check(self._lib.fca_context_dims(self._h, ctypes.byref(n), ctypes.byref(m)),
                    "fca_context_dims")
        return int(n.value), int(m.value)

    def copy_layout(self, which: str) -> np.ndarray:
        """Host copy of the device ``rows``, ``cols`` (padded to 4-word rows) or ``top`` in processing
        order, or the processing ``order`` (position of each attribute)."""
        wn = words(self.n_objects)
        wnp = (wn + 3) & ~3
        shape = {"rows": (self.n_objects, self.wm), "cols": (self.n_attrs, wnp), "top": (self.wm,),
                 "order": (self.n_attrs,)}[which]
        dst = np.zeros(shape, dtype=np.uint32)
        code = {"rows": 0, "cols": 1, "top": 2, "order": 3}[which]
        self._check(self._lib.fca_context_copy(self._h, code, ctypes.c_void_p(dst.ctypes.data), dst.size),
                    "fca_context_copy")
        return dst


def enumerate_intents(rows: np.ndarray, n_objects: int, n_attrs: int) -> np.ndarray:
    """Convenience: all intents of a host context as a host ``(K, W_M)`` uint32 array."""
    with Context(rows, n_objects, n_attrs) as ctx:
        out = ctx.enumerate()
        return out.cpu().numpy().view(np.uint32)
