"""GPU parity of the lattice calls (fca_extents, fca_cover_edges) against the CPU oracle.

The inputs are the oracle's own intents. Extents must equal the oracle's (the extents its search
keeps, and Y' from the derivation operator), word for word. Cover edges must equal the oracle's
cover relation as a set of (upper row, lower row) pairs. At the full sparse size they are checked
by properties of a Hasse diagram plus the lower covers of sampled concepts. Both processing orders
of the context are covered: the rows the kernels read are permuted under the support order.
"""
import numpy as np
import pytest

import oracle
from oracle import lattice
from closed_set_enumeration_gb300 import build as fbuild
from closed_set_enumeration_gb300 import contexts as cx
from tests._util import attrs_to_row

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fbuild.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).cuda()


def host(t):
    return t.cpu().numpy().view(np.uint32)


def chain(n):
    return cx.pack_rows(np.tril(np.ones((n, n), dtype=bool)))


# shapes straddle the word boundaries of objects and attributes and the 64-object switch of the
# cover kernel (its extents of at most 64 objects are 64-bit masks, larger ones object bitmaps; the
# cover cases of 2 100 and 5 000 objects give compacted sub-extents of more than 32 and 128 words)
EXT_CASES = [(1, 1, 0.5, 0), (31, 7, 0.3, 1), (33, 31, 0.3, 2), (64, 65, 0.12, 3), (65, 20, 0.3, 4),
             (130, 64, 0.12, 5), (257, 45, 0.2, 6), (1500, 40, 0.12, 7), (600, 96, 0.12, 8), (40, 1000, 0.02, 9)]


@pytest.mark.parametrize("order", ["0", "2"])
@pytest.mark.parametrize("n,m,p,seed", EXT_CASES)
def test_extents_match_oracle(n, m, p, seed, order, monkeypatch):
    monkeypatch.setenv("FCA_ATTR_ORDER", order)
    from closed_set_enumeration_gb300 import fca
    rows = cx.random_context(n, m, p, seed)
    ref = oracle.cbo(rows, n, m, want_extents=True)
    with fca.Context(rows, n, m) as ctx:
        got = host(ctx.extents(dev(ref["intents"])))
        torch.cuda.synchronize()
    assert got.shape == ref["extents"].shape
    assert np.array_equal(got, ref["extents"])
    pick = np.random.default_rng(seed).choice(got.shape[0], min(50, got.shape[0]), replace=False)
    for i in pick:
        want = cx.pack_rows(oracle.derive_extent(rows, ref["intents"][i])[None, :])[0]
        assert np.array_equal(got[i], want)


def test_extents_edge_cases():
    from closed_set_enumeration_gb300 import fca
    n, m = 70, 40
    rows = cx.random_context(n, m, 0.5, 3)
    sets = [attrs_to_row([], m), attrs_to_row(range(m), m), attrs_to_row([0], m), attrs_to_row([39], m),
            attrs_to_row([3, 17, 33], m)]
    x = np.stack(sets)
    noisy = x.copy()
    noisy[:, -1] |= np.uint32(0xffffffff) << np.uint32(m & 31)   # padding bits past M set
    with fca.Context(rows, n, m) as ctx:
        empty = ctx.extents(dev(np.zeros((0, 2), np.uint32)))
        assert tuple(empty.shape) == (0, 3)
        a = host(ctx.extents(dev(x)))
        b = host(ctx.extents(dev(noisy)))
    assert np.array_equal(a, b)
    for i in range(x.shape[0]):
        want = cx.pack_rows(oracle.derive_extent(rows, x[i])[None, :])[0]
        assert np.array_equal(a[i], want)
    assert a[0].tolist() == [0xffffffff, 0xffffffff, (1 << 6) - 1]   # every object, padding clear


def test_extents_full_size_sparse():
    """All 149 629 concepts of the sparse workload (2 000 x 64): every extent against the oracle's."""
    from closed_set_enumeration_gb300 import fca
    w = cx.WORKLOADS["sparse"]
    rows = w.rows()
    ref = oracle.cbo(rows, w.n_objects, w.n_attrs, threads=8, want_extents=True)
    with fca.Context(rows, w.n_objects, w.n_attrs) as ctx:
        got = host(ctx.extents(dev(ref["intents"])))
    assert np.array_equal(got, ref["extents"])


def gpu_covers(rows, n, m, intents, capacity=None):
    from closed_set_enumeration_gb300 import fca
    with fca.Context(rows, n, m) as ctx:
        e = ctx.cover_edges(dev(intents), capacity=capacity)
        return host(e).astype(np.int64).reshape(-1, 2)


def edge_set(e):
    return sorted(map(tuple, np.asarray(e, dtype=np.int64).tolist()))


COVER_CASES = [("contranominal", 10), ("identity", 40), ("chain", 33), ("random", (60, 12, 0.35, 5)),
               ("random", (100, 20, 0.2, 6)), ("random", (200, 40, 0.15, 7)), ("random", (64, 33, 0.3, 8)),
               ("random", (65, 70, 0.12, 9)), ("random", (300, 45, 0.1, 10)), ("random", (1000, 30, 0.1, 11)),
               ("random", (40, 1000, 0.02, 9)), ("random", (2100, 28, 0.1, 14)), ("random", (5000, 16, 0.15, 12)),
               ("divisors", (5000, 24))]


def cover_context(kind, arg):
    if kind == "contranominal":
        return cx.contranominal(arg), arg, arg
    if kind == "identity":
        return cx.identity(arg), arg, arg
    if kind == "chain":
        return chain(arg), arg, arg
    if kind == "divisors":
        # object o (1..n) has attribute a when a + 1 divides o: nested columns (the multiples of 4 lie
        # inside the multiples of 2) spread over every word of the object bitmap, so containment tests
        # of large extents run to the last word
        n, m = arg
        o = np.arange(1, n + 1)[:, None]
        return cx.pack_rows(o % np.arange(2, m + 2)[None, :] == 0), n, m
    n, m, p, s = arg
    return cx.random_context(n, m, p, s), n, m


@pytest.mark.parametrize("order", ["0", "2"])
@pytest.mark.parametrize("kind,arg", COVER_CASES)
def test_cover_edges_match_oracle(kind, arg, order, monkeypatch):
    monkeypatch.setenv("FCA_ATTR_ORDER", order)
    rows, n, m = cover_context(kind, arg)
    intents = oracle.cbo(rows, n, m)["intents"]
    want = edge_set(lattice.cover_edges(intents, m))
    got = gpu_covers(rows, n, m, intents)
    assert len(got) == len(want)
    assert edge_set(got) == want
    # any row order of the input: the edges follow the rows
    perm = np.random.default_rng(1).permutation(intents.shape[0])
    got2 = gpu_covers(rows, n, m, intents[perm])
    assert edge_set(perm[got2]) == want


def test_cover_edges_capacity_and_incomplete_set():
    from closed_set_enumeration_gb300 import fca
    rows, n, m = cx.contranominal(6), 6, 6
    intents = oracle.cbo(rows, n, m)["intents"]
    want = set(edge_set(lattice.cover_edges(intents, m)))
    with fca.Context(rows, n, m) as ctx:
        buf = torch.zeros((10, 2), dtype=torch.int32, device="cuda")
        st, count = ctx.cover_edges_into(dev(intents), buf)
        assert st == fca.FCA_ERR_CAPACITY and count == len(want) == 6 * 2 ** 5
        assert set(edge_set(host(buf).astype(np.int64))) <= want
        st0, count0 = ctx.cover_edges_into(dev(intents), buf, capacity=0)
        assert st0 == fca.FCA_ERR_CAPACITY and count0 == count
        # the bottom intent (every attribute) left out: its upper neighbours find no row for it
        sizes = cx.unpack_rows(intents, m).sum(axis=1)
        missing = intents[sizes < m]
        with pytest.raises(fca.FcaError) as err:
            ctx.cover_edges(dev(missing))
        assert err.value.status == fca.FCA_ERR_INVALID


@pytest.mark.parametrize("dup_row,padding", [(0, False), (17, False), (17, True)])
def test_cover_edges_reject_a_repeated_intent(dup_row, padding):
    """An intent given twice (also when the copy differs only in padding bits past M, which are
    ignored) is refused with FCA_ERR_INVALID instead of edges that resolve to either copy; the same
    set without the copy is accepted."""
    from closed_set_enumeration_gb300 import fca
    rows, n, m = cx.random_context(90, 37, 0.2, 3), 90, 37
    intents = oracle.cbo(rows, n, m)["intents"]
    copy = intents[dup_row].copy()
    if padding:
        copy[-1] |= np.uint32(1 << 31)   # bit 63: past M = 37
    with fca.Context(rows, n, m) as ctx:
        with pytest.raises(fca.FcaError) as err:
            ctx.cover_edges(dev(np.vstack([intents, copy[None, :]])))
        assert err.value.status == fca.FCA_ERR_INVALID
        assert "repeat" in str(err.value)
        e = host(ctx.cover_edges(dev(intents))).astype(np.int64).reshape(-1, 2)
        assert edge_set(e) == edge_set(lattice.cover_edges(intents, m))


@pytest.mark.parametrize("order", ["0", "2"])
def test_cover_edges_full_size_sparse(order, monkeypatch):
    """The sparse workload (2 000 x 64, 149 629 concepts): Hasse-diagram properties on every edge,
    and the lower covers of sampled concepts (with the top and the bottom) against the oracle."""
    monkeypatch.setenv("FCA_ATTR_ORDER", order)
    w = cx.WORKLOADS["sparse"]
    rows = w.rows()
    m = w.n_attrs
    intents = oracle.cbo(rows, w.n_objects, m, threads=8)["intents"]
    k = intents.shape[0]
    e = gpu_covers(rows, w.n_objects, m, intents)
    assert np.unique(e[:, 0] * k + e[:, 1]).size == e.shape[0]          # no edge twice
    up, lo = intents[e[:, 0]], intents[e[:, 1]]
    assert np.all((up & lo) == up) and not np.any(np.all(up == lo, axis=1))   # proper inclusion
    sizes = cx.unpack_rows(intents, m).sum(axis=1)
    has_up = np.zeros(k, bool)
    has_down = np.zeros(k, bool)
    has_up[e[:, 1]] = True
    has_down[e[:, 0]] = True
    top, bottom = int(np.argmin(sizes)), int(np.argmax(sizes))
    assert has_up.sum() == k - 1 and not has_up[top]
    assert has_down.sum() == k - 1 and not has_down[bottom]
    order_e = np.argsort(e[:, 0], kind="stable")
    starts = np.searchsorted(e[order_e, 0], np.arange(k + 1))
    pick = list(np.random.default_rng(5).choice(k, 150, replace=False)) + [top, bottom]
    for i in pick:
        mine = np.sort(e[order_e[starts[i]:starts[i + 1]], 1])
        assert mine.tolist() == lattice.lower_covers_of(intents, m, int(i)).tolist(), i


def test_pool_options_via_set_option():
    """Pool sizes set through fca_set_option (not the environment) still give the oracle's set."""
    from closed_set_enumeration_gb300 import fca
    n, m = 1500, 40
    rows = cx.random_context(n, m, 0.3, 1)
    ref = oracle.cbo(rows, n, m)["intents"]
    with fca.Context(rows, n, m) as ctx:
        ctx.set_option(fca.FCA_OPT_LEVEL_BYTES, 1 << 16)
        ctx.set_option(fca.FCA_OPT_QUEUE_ENTRIES, 256)
        got = host(ctx.enumerate()).reshape(-1, 2)
        for bad in ((fca.FCA_OPT_ATTR_ORDER, 3), (fca.FCA_OPT_LEVEL_BYTES, -1), (99, 1)):
            with pytest.raises(fca.FcaError):
                ctx.set_option(*bad)
    assert got.shape == ref.shape
    assert np.array_equal(np.unique(got, axis=0), np.unique(ref, axis=0))
