"""Host-side checks of the C ABI: the library loads, exports every declared entry
point, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

from closed_set_enumeration_gb300 import build as fbuild
from closed_set_enumeration_gb300 import fca

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fca.h")


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fca.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fca_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(fca.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert fca.status_string(fca.FCA_OK) == "ok"
    assert fca.status_string(fca.FCA_ERR_CAPACITY) == "capacity exceeded"
    assert fca.status_string(99) == "unknown status"


def test_create_rejects_bad_arguments_without_gpu_work(lib):
    h = ctypes.c_void_p(123)
    rows = np.zeros((4, 1), dtype=np.uint32)
    p = ctypes.c_void_p(rows.ctypes.data)
    assert lib.fca_context_create(None, 4, 5, ctypes.byref(h)) == fca.FCA_ERR_INVALID
    assert not h.value
    assert lib.fca_context_create(p, 0, 5, ctypes.byref(h)) == fca.FCA_ERR_INVALID
    assert lib.fca_context_create(p, 4, 0, ctypes.byref(h)) == fca.FCA_ERR_INVALID
    assert lib.fca_context_create(p, 4, 1025, ctypes.byref(h)) == fca.FCA_ERR_INVALID
    assert lib.fca_context_create(p, 4, 5, None) == fca.FCA_ERR_INVALID


def test_null_context_calls(lib):
    cnt = ctypes.c_uint64(0)
    assert lib.fca_enumerate(None, None, 0, ctypes.byref(cnt), None) == fca.FCA_ERR_INVALID
    assert lib.fca_enumerate_host(None, None, 0, ctypes.byref(cnt), None) == fca.FCA_ERR_INVALID
    assert lib.fca_extents(None, None, 0, None, None) == fca.FCA_ERR_INVALID
    assert lib.fca_cover_edges(None, None, 0, None, 0, ctypes.byref(cnt), None) == fca.FCA_ERR_INVALID
    s = fca.FcaStats()
    assert lib.fca_get_stats(None, ctypes.byref(s)) == fca.FCA_ERR_INVALID
    assert lib.fca_last_error(None) == b""
    lib.fca_free(None)   # NULL is ignored


def test_binding_constants_match_the_header():
    """The binding's status and option numbers are the header's enum values."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    values = {k: int(v) for k, v in re.findall(r"\b(FCA_[A-Z_0-9]+)\s*=\s*(\d+)", text)}
    assert values["FCA_OPT_WAIT_LIMIT_NS"] == 6
    for name, v in values.items():
        assert getattr(fca, name) == v, name
