"""The allocation-free entry point, for callers that may not call cudaMalloc while they run.

fca_enumerate_small_noalloc keeps all of its scratch in one device array of the
library and allocates nothing; its result must equal fca_enumerate's exactly
(the same intent set) on two calls in a row, which also checks that a call
starts from a clean scratch array whatever the previous call left in it.
This file is collected last so that a failure here cannot hide other tests.
"""
import ctypes

import numpy as np
import pytest

from closed_set_enumeration_gb300 import build as fbuild
from closed_set_enumeration_gb300 import contexts as cx
from tests._util import same_set

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def _noalloc(lib, rows, n, m, capacity):
    wm = (m + 31) // 32
    dev_rows = torch.from_numpy(np.ascontiguousarray(rows).view(np.int32)).cuda()
    out = torch.full((max(capacity, 1), wm), -1, dtype=torch.int32, device="cuda")
    count = ctypes.c_uint64(0)
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.fca_enumerate_small_noalloc(ctypes.c_void_p(dev_rows.data_ptr()), n, m,
                                         ctypes.c_void_p(out.data_ptr()), capacity, ctypes.byref(count),
                                         ctypes.c_void_p(stream))
    return st, int(count.value), out[: int(count.value)].cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("n,m,density,seed", [(64, 16, 0.3, 0), (20, 70, 0.4, 1), (64, 1024, 0.1, 2),
                                              (33, 33, 0.35, 3), (1, 5, 0.5, 4)])
def test_noalloc_matches_enumerate_twice(lib, n, m, density, seed):
    rows = cx.WORKLOADS["tiny"].rows() if seed == 0 else cx.random_context(n, m, density, seed)
    ref = _reference(rows, n, m)
    for _ in range(2):
        st, cnt, got = _noalloc(lib, rows, n, m, ref.shape[0] + 3)
        assert st == 0 and cnt == ref.shape[0]
        assert same_set(got, ref)


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
