"""The allocation-free entry point, for callers that may not call cudaMalloc while they run.

fca_enumerate_small_noalloc keeps all of its scratch in one device array of the
library and allocates nothing. Its result must equal fca_enumerate's exactly
(the same intent set) and the CPU oracle's, on two calls in a row, which also
checks that a call starts from a clean scratch array whatever the previous call
left in it. The capacity contract is checked as for fca_enumerate: a short
buffer receives only true intents, no row past its end is written and the
count stays exact. This file is collected last so that a failure here cannot
hide other tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
from closed_set_enumeration_gb300 import build as fbuild
from closed_set_enumeration_gb300 import contexts as cx
from tests._util import has_duplicates, same_set, sort_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SENTINEL = -1   # 0xffffffff in every word: a row no intent of these contexts can equal (padding bits)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fbuild.build()
    from closed_set_enumeration_gb300 import fca
    return fca.load_library()


def _reference(rows, n, m):
    from closed_set_enumeration_gb300 import fca
    with fca.Context(rows, n, m) as ctx:
        return ctx.enumerate().cpu().numpy().view(np.uint32)


def _noalloc(lib, rows, n, m, capacity, buffer_rows=None):
    """Call the entry point on device rows; returns (status, count, rows written, whole buffer)."""
    wm = (m + 31) // 32
    dev_rows = torch.from_numpy(np.ascontiguousarray(rows).view(np.int32)).cuda()
    size = max(capacity, 1) if buffer_rows is None else buffer_rows
    out = torch.full((size, wm), SENTINEL, dtype=torch.int32, device="cuda")
    count = ctypes.c_uint64(0)
    stream = torch.cuda.current_stream().cuda_stream
    ptr = out.data_ptr() if capacity > 0 else 0
    st = lib.fca_enumerate_small_noalloc(ctypes.c_void_p(dev_rows.data_ptr()), n, m, ctypes.c_void_p(ptr),
                                         capacity, ctypes.byref(count), ctypes.c_void_p(stream))
    torch.cuda.synchronize()
    whole = out.cpu().numpy().view(np.uint32)
    k = min(int(count.value), capacity)
    return st, int(count.value), whole[:k], whole


@pytest.mark.parametrize("n,m,density,seed", [(64, 16, 0.3, 0), (20, 70, 0.4, 1), (64, 1024, 0.1, 2),
                                              (33, 33, 0.35, 3), (1, 5, 0.5, 4)])
def test_noalloc_matches_enumerate_and_oracle_twice(lib, n, m, density, seed):
    rows = cx.WORKLOADS["tiny"].rows() if seed == 0 else cx.random_context(n, m, density, seed)
    ref = _reference(rows, n, m)
    want = oracle.cbo(rows, n, m)["intents"]
    assert same_set(ref, want)
    for _ in range(2):
        st, cnt, got, _ = _noalloc(lib, rows, n, m, ref.shape[0] + 3)
        assert st == 0 and cnt == ref.shape[0]
        assert same_set(got, ref)
        assert same_set(got, want)


def _full_row_context(n, m, seed, full):
    rows = cx.random_context(n, m, 0.3, seed)
    wm = (m + 31) // 32
    for o in range(n):        # no object holds every attribute ...
        rows[o, 0] &= ~np.uint32(1)
    if full:                  # ... except, in the second case, one object that holds them all
        rows[n // 2] = 0xFFFFFFFF
        if m % 32:
            rows[n // 2, wm - 1] = (1 << (m % 32)) - 1
    return rows


@pytest.mark.parametrize("full", [False, True])
def test_noalloc_bottom_concept(lib, full):
    """The bottom intent (every attribute) is output once in both of its cases: appended by the
    host when no object holds every attribute (its extent is empty), found by the search when
    one object does."""
    n, m = 40, 45
    rows = _full_row_context(n, m, 7, full)
    want = oracle.cbo(rows, n, m)["intents"]
    bottom = cx.pack_rows(np.ones((1, m), dtype=bool))[0]
    assert (want == bottom).all(axis=1).sum() == 1
    for _ in range(2):
        st, cnt, got, _ = _noalloc(lib, rows, n, m, want.shape[0])
        assert st == 0 and cnt == want.shape[0]
        assert same_set(got, want)


@pytest.mark.parametrize("full", [False, True])
def test_noalloc_capacity_contract(lib, full):
    """capacity 0 (out NULL), 1 and count - 1: status FCA_ERR_CAPACITY with the exact count, only
    true intents in the rows written, none twice, and no row past the capacity touched."""
    n, m = 50, 37
    rows = _full_row_context(n, m, 11, full)
    want = oracle.cbo(rows, n, m)["intents"]
    total = want.shape[0]
    want_set = {tuple(r) for r in sort_rows(want)}
    top = oracle.derive_intent(rows, np.ones(n, dtype=bool), m)
    for cap in (0, 1, total - 1):
        st, cnt, got, whole = _noalloc(lib, rows, n, m, cap, buffer_rows=cap + 4)
        assert st == 3 and cnt == total        # FCA_ERR_CAPACITY, exact count
        assert got.shape[0] == cap
        assert all(tuple(r) in want_set for r in got)
        assert not has_duplicates(got)
        if cap >= 1:
            assert np.array_equal(got[0], top)  # the top intent is row 0
        assert (whole[cap:] == np.uint32(0xFFFFFFFF)).all()
    st, cnt, got, _ = _noalloc(lib, rows, n, m, total)
    assert st == 0 and cnt == total and same_set(got, want)


def test_noalloc_rejects_sizes_beyond_its_limit(lib):
    rows = cx.random_context(65, 8, 0.3, 0)
    count = ctypes.c_uint64(0)
    out = torch.empty((8, 1), dtype=torch.int32, device="cuda")
    st = lib.fca_enumerate_small_noalloc(ctypes.c_void_p(rows.ctypes.data), 65, 8,
                                         ctypes.c_void_p(out.data_ptr()), 8, ctypes.byref(count), None)
    assert st == 1   # FCA_ERR_INVALID
    rows = cx.random_context(10, 8, 0.3, 0)
    st = lib.fca_enumerate_small_noalloc(ctypes.c_void_p(rows.ctypes.data), 10, 1025,
                                         ctypes.c_void_p(out.data_ptr()), 8, ctypes.byref(count), None)
    assert st == 1
