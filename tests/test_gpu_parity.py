"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

The intent set must be bit-exact (compared as a sorted set; output order is
unspecified), the number of closures evaluated must equal the oracle's over the
table in the same processing order (ascending support by default), and no
intent may appear twice.
"""
import json
import os

import numpy as np
import pytest

import oracle
from closed_set_enumeration_gb300 import build as fbuild
from closed_set_enumeration_gb300 import contexts as cx
from tests._util import (GOLDEN, attrs_to_row, golden_names, has_duplicates, load_golden,
                         same_set, sort_rows, support_order)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fbuild.build()


def gpu_run(rows, n, m, capacity=None):
    from closed_set_enumeration_gb300 import fca
    with fca.Context(rows, n, m) as ctx:
        out = ctx.enumerate(capacity=capacity)
        got = out.cpu().numpy().view(np.uint32).reshape(-1, (m + 31) // 32)
        return got, ctx.stats()


def ordered_closures(rows, n, m, threads=1):
    """The oracle's closures over the table in the library's default processing order."""
    return oracle.cbo(support_order(rows, n, m)[0], n, m, threads=threads)["closures"]


def check_against_oracle(rows, n, m, threads=1):
    got, st = gpu_run(rows, n, m)
    ref = oracle.cbo(rows, n, m, threads=threads)
    assert not has_duplicates(got)
    assert same_set(got, ref["intents"])
    assert st["concepts"] == ref["intents"].shape[0]
    assert st["closures"] == ordered_closures(rows, n, m, threads)
    return got, st


@pytest.mark.parametrize("name", golden_names())
def test_golden(name):
    n, m, rows, expected = load_golden(name)
    got, _ = gpu_run(rows, n, m)
    assert same_set(got, expected)


# shapes straddle the word and tier boundaries (32 / 64 objects, 32 / 64 attributes); the
# densities keep each oracle run well under a second (denser tables explode combinatorially)
CASES = [(n, m, d, s)
         for (n, m) in [(1, 1), (1, 40), (2, 3), (31, 7), (32, 33), (33, 31), (63, 64), (64, 65),
                        (65, 20), (96, 100), (130, 64), (257, 45), (1500, 40)]
         for (d, s) in [(0.12, 0), (0.3, 1)]] + [(600, 96, 0.12, 0), (600, 96, 0.2, 1)]


@pytest.mark.parametrize("n,m,density,seed", CASES)
def test_random_contexts(n, m, density, seed):
    rows = cx.random_context(n, m, density, seed)
    check_against_oracle(rows, n, m)


@pytest.mark.parametrize("n,m,density,seed", [(3000, 128, 0.08, 3), (2000, 300, 0.03, 4),
                                              (5000, 1024, 0.004, 5), (800, 1000, 0.02, 6),
                                              # 100-256 objects with many attributes: bitmap-tier roots,
                                              # subtrees with many relevant attributes (shared-memory path)
                                              (250, 300, 0.1, 2), (200, 128, 0.15, 3), (256, 200, 0.12, 4),
                                              (120, 300, 0.2, 5), (100, 700, 0.1, 6),
                                              # parents above and below the restricted-column limit:
                                              # both paths of the bitmap tier
                                              (9000, 24, 0.25, 2), (12000, 40, 0.2, 3)])
def test_larger_random_contexts(n, m, density, seed):
    rows = cx.random_context(n, m, density, seed)
    check_against_oracle(rows, n, m, threads=8)


@pytest.mark.parametrize("n", [5, 16, 20])
def test_contranominal(n):
    got, st = gpu_run(cx.contranominal(n), n, n)
    assert got.shape[0] == 2 ** n and not has_duplicates(got)
    assert st["closures"] == 2 ** n - 1


@pytest.mark.parametrize("n", [2, 33, 64, 65, 200, 1024])
def test_identity(n):
    got, st = gpu_run(cx.identity(n), n, n)
    expected = [attrs_to_row([], n), attrs_to_row(range(n), n)] + [attrs_to_row([j], n) for j in range(n)]
    assert same_set(got, np.stack(expected))
    assert st["closures"] == n + n * (n - 1) // 2


@pytest.mark.parametrize("n,m", [(1, 1), (40, 33), (70, 64), (100, 100)])
def test_all_zero_and_all_ones(n, m):
    w = (m + 31) // 32
    zero = np.zeros((n, w), dtype=np.uint32)
    got, st = gpu_run(zero, n, m)
    assert same_set(got, np.stack([attrs_to_row([], m), attrs_to_row(range(m), m)]))
    assert st["closures"] == m
    ones = np.tile(attrs_to_row(range(m), m), (n, 1))
    got, st = gpu_run(ones, n, m)
    assert same_set(got, attrs_to_row(range(m), m)[None, :])
    assert st["closures"] == 0


def test_full_row_object_reaches_bottom_through_search():
    # one object holds every attribute, so the bottom concept has a non-empty extent
    rows = cx.random_context(300, 70, 0.2, 9)
    rows[17] = attrs_to_row(range(70), 70)
    check_against_oracle(rows, 300, 70)


def test_padding_bits_ignored():
    rows = cx.random_context(200, 37, 0.3, 2)
    dirty = rows.copy()
    dirty[:, -1] |= np.uint32(0xFFFFFFE0)
    got, _ = gpu_run(dirty, 200, 37)
    assert same_set(got, oracle.cbo(rows, 200, 37)["intents"])
    assert not np.any(got[:, -1] & np.uint32(0xFFFFFFE0))


def test_device_rows_input():
    from closed_set_enumeration_gb300 import fca
    rows = cx.random_context(500, 50, 0.2, 4)
    dev = torch.from_numpy(rows.view(np.int32)).cuda()
    with fca.Context(dev, 500, 50) as ctx:
        got = ctx.enumerate().cpu().numpy().view(np.uint32)
        assert np.array_equal(ctx.copy_layout("rows"), support_order(rows, 500, 50)[0])
    assert same_set(got, oracle.cbo(rows, 500, 50)["intents"])


@pytest.mark.parametrize("order", ["0", "1", "2"])
def test_column_layout_is_transpose(monkeypatch, order):
    # the device tables in processing order: attribute order (0), or ascending support (2, and 1
    # for this table, whose supports vary)
    from closed_set_enumeration_gb300 import fca
    monkeypatch.setenv("FCA_ATTR_ORDER", order)
    n, m = 1000, 70
    rows = cx.random_context(n, m, 0.3, 1)
    rows[:, 0] |= np.uint32(0x0000F00F)    # uneven supports among the first attributes
    prows, inv = support_order(rows, n, m) if order != "0" else (rows, np.arange(m))
    with fca.Context(rows, n, m) as ctx:
        cols = ctx.copy_layout("cols")
        top = ctx.copy_layout("top")
        pos = ctx.copy_layout("order")
        got = ctx.enumerate().cpu().numpy().view(np.uint32).reshape(-1, (m + 31) // 32)
        st = ctx.stats()
    cells = cx.unpack_rows(prows, m)
    wn = (n + 31) // 32
    expect = cx.pack_rows(cells.T)
    assert np.array_equal(pos[inv], np.arange(m))
    assert np.array_equal(cols[:, :wn], expect)
    assert not np.any(cols[:, wn:])
    assert np.array_equal(top, oracle.derive_intent(prows, np.ones(n, bool), m))
    # the output is in attribute order either way; the closures follow the processing order
    assert same_set(got, oracle.cbo(rows, n, m, threads=8)["intents"])
    assert st["closures"] == oracle.cbo(prows, n, m, threads=8)["closures"]


def test_capacity_contract():
    from closed_set_enumeration_gb300 import fca
    rows = cx.random_context(300, 40, 0.3, 5)
    ref = oracle.cbo(rows, 300, 40)["intents"]
    total = ref.shape[0]
    with fca.Context(rows, 300, 40) as ctx:
        st, cnt = ctx.enumerate_into(torch.empty((0, 2), dtype=torch.int32, device="cuda"), 0)
        assert st == fca.FCA_ERR_CAPACITY and cnt == total
        small = torch.full((10, 2), -1, dtype=torch.int32, device="cuda")
        st, cnt = ctx.enumerate_into(small, 10)
        assert st == fca.FCA_ERR_CAPACITY and cnt == total
        part = small.cpu().numpy().view(np.uint32)
        refset = set(map(tuple, ref))
        assert all(tuple(r) in refset for r in part)           # only true intents written
        assert np.array_equal(part[0], oracle.derive_intent(rows, np.ones(300, bool), 40))
        exact = torch.empty((total, 2), dtype=torch.int32, device="cuda")
        st, cnt = ctx.enumerate_into(exact, total)
        assert st == fca.FCA_OK and cnt == total
        assert same_set(exact.cpu().numpy().view(np.uint32), ref)


def test_enumerate_host_and_reuse():
    from closed_set_enumeration_gb300 import fca
    rows = cx.random_context(400, 64, 0.25, 8)
    ref = oracle.cbo(rows, 400, 64)["intents"]
    with fca.Context(rows, 400, 64) as ctx:
        host = np.zeros((ref.shape[0] + 5, 2), dtype=np.uint32)
        st, cnt = ctx.enumerate_host(host)
        assert st == fca.FCA_OK and cnt == ref.shape[0]
        assert same_set(host[:cnt], ref)
        for _ in range(2):   # pools are reused across calls
            got = ctx.enumerate().cpu().numpy().view(np.uint32)
            assert same_set(got, ref)


def test_default_order_keeps_attribute_order_on_even_supports(monkeypatch):
    # option 1 (the default): on a table whose supports hardly vary the search keeps attribute
    # order, and its closures are the oracle's in attribute order
    from closed_set_enumeration_gb300 import fca
    monkeypatch.setenv("FCA_ATTR_ORDER", "1")
    n, m = 2000, 64
    rows = cx.random_context(n, m, 0.15, 1)
    ref = oracle.cbo(rows, n, m, threads=8)
    with fca.Context(rows, n, m) as ctx:
        assert np.array_equal(ctx.copy_layout("order"), np.arange(m))
        got = ctx.enumerate(capacity=ref["intents"].shape[0] + 1).cpu().numpy().view(np.uint32).reshape(-1, 2)
        st = ctx.stats()
    assert same_set(got, ref["intents"])
    assert st["closures"] == ref["closures"]


@pytest.mark.parametrize("pregrow", ["0", "1"])
@pytest.mark.parametrize("limit", [None, "1"])
def test_small_pools_roll_back_and_chunk(monkeypatch, limit, pregrow):
    # tiny initial pools: launches overflow, are rolled back and retried after the destinations are
    # emptied or grown; with a 1-byte growth limit, levels are split into ever smaller chunks instead.
    # With growth ahead of the launches (pregrow 1) the same output must come whichever path runs.
    n, m = 4000, 60
    rows = cx.random_context(n, m, 0.12, 12)
    rows[: n // 4, 0] |= np.uint32(0x00FF00FF)      # dense block -> large extents and deep bitmap levels
    ref = oracle.cbo(rows, n, m, threads=8)
    monkeypatch.setenv("FCA_LEVEL_BYTES", "1")       # floor: 4*M entries per level
    monkeypatch.setenv("FCA_QUEUE_ENTRIES", "1")     # floor: 4*M entries per queue
    monkeypatch.setenv("FCA_PREGROW", pregrow)
    if limit:
        monkeypatch.setenv("FCA_POOL_LIMIT_BYTES", limit)
    # output sized up front: a capacity miss would re-run the enumeration on the pools the first
    # run grew, and the statistics would describe that second run
    got, st = gpu_run(rows, n, m, capacity=ref["intents"].shape[0] + 1)
    assert not has_duplicates(got)
    assert same_set(got, ref["intents"])
    assert st["closures"] == ordered_closures(rows, n, m, threads=8)
    if pregrow == "0" or limit:
        assert st["retries"] > 0


def test_chained_levels_roll_back(monkeypatch):
    # After a first call, bitmap levels are launched as one chain as deep as that call's search.
    # A second table of the same shape with a deeper, larger search overflows the (tiny) pools
    # inside such a chain: the chain is committed up to the launch that overflowed, which is rolled
    # back and retried launch by launch; a third call on the same table then chains without
    # overflowing.
    from closed_set_enumeration_gb300 import fca
    n, m = 4000, 60
    rows_a = cx.random_context(n, m, 0.10, 21)
    rows_a[: n // 5, 0] |= np.uint32(0x000F000F)
    rows_b = cx.random_context(n, m, 0.12, 22)
    rows_b[: n // 3, 0] |= np.uint32(0x00FF00FF)
    ref_a = oracle.cbo(rows_a, n, m, threads=8)
    ref_b = oracle.cbo(rows_b, n, m, threads=8)
    monkeypatch.setenv("FCA_LEVEL_BYTES", "1")
    monkeypatch.setenv("FCA_QUEUE_ENTRIES", "1")
    monkeypatch.setenv("FCA_PREGROW", "0")
    wm = (m + 31) // 32
    with fca.Context(rows_a, n, m) as ctx:
        got = ctx.enumerate(capacity=ref_a["intents"].shape[0] + 1).cpu().numpy().view(np.uint32).reshape(-1, wm)
        assert same_set(got, ref_a["intents"])
        assert ctx.stats()["levels"] >= 4
        ctx.load(rows_b)
        retries = []
        for _ in range(2):
            got = ctx.enumerate(capacity=ref_b["intents"].shape[0] + 1).cpu().numpy().view(np.uint32).reshape(-1, wm)
            st = ctx.stats()
            retries.append(st["retries"])
            assert not has_duplicates(got)
            assert same_set(got, ref_b["intents"])
            assert st["closures"] == ordered_closures(rows_b, n, m, threads=8)
        # the second table's first call overflowed, the last one reused the grown pools
        assert retries[0] > 0 and retries[1] == 0


@pytest.mark.parametrize("name", ["tiny", "sparse"])
def test_workload_full_set(name):
    w = cx.WORKLOADS[name]
    check_against_oracle(w.rows(), w.n_objects, w.n_attrs, threads=8)


DIGESTS = os.path.join(GOLDEN, "workload_digests.json")


def _digest(intents):
    import hashlib
    rows = sort_rows(np.ascontiguousarray(intents, dtype="<u4"))
    return hashlib.sha256(np.ascontiguousarray(rows).tobytes()).hexdigest()


@pytest.mark.parametrize("name", ["sparse", "skewed", "zipf", "biclusters_50k", "biclusters"])
def test_workload_full_size_digest(name):
    """Full-size workloads against oracle digests written by tests/golden/make_workload_digests.py:
    exact count and closures (in the processing order of the tests), the order-independent
    multiset digest of the intent set and the SHA-256 of the sorted set where recorded, and fixed
    points B'' = B of sampled intents computed one by one by the oracle's derivation operators."""
    from tests._util import multiset_digest
    table = json.load(open(DIGESTS)) if os.path.exists(DIGESTS) else {}
    if name not in table:
        pytest.skip(f"no oracle digest stored for {name}")
    ref = table[name]
    w = cx.WORKLOADS[name]
    rows = w.rows()
    got, st = gpu_run(rows, w.n_objects, w.n_attrs, capacity=ref["concepts"])
    assert got.shape[0] == ref["concepts"]
    assert st["closures"] == ref["closures_support_order"]   # the default processing order
    if "multiset_hsum" in ref:
        assert multiset_digest(got) == (int(ref["multiset_hsum"], 16), int(ref["multiset_hxor"], 16))
    if "sha256_sorted_intents" in ref:
        assert _digest(got) == ref["sha256_sorted_intents"]
    rng = np.random.default_rng(0)
    for i in rng.choice(got.shape[0], 200, replace=False):
        ext = oracle.derive_extent(rows, got[i])
        assert np.array_equal(oracle.derive_intent(rows, ext, w.n_attrs), got[i])


def test_bounded_wait_reports_instead_of_hanging():
    """The object-list kernel's work-sharing wait is bounded (FCA_OPT_WAIT_LIMIT_NS). A single
    object-list root (contranominal scale of 20 objects: one subtree of 2^20 concepts) is split
    into slices, and the warps whose slices are empty wait for hand-overs from the busy ones. With
    the limit at 1 ns their waits run out: the call must return FCA_ERR_CUDA with the wait message
    (no hang, no device fault), and the same context must then enumerate correctly with the
    default limit."""
    from closed_set_enumeration_gb300 import fca
    n = 20
    rows = cx.contranominal(n)
    want = oracle.cbo(rows, n, n)["intents"]
    with fca.Context(rows, n, n) as ctx:
        ctx.set_option(fca.FCA_OPT_WAIT_LIMIT_NS, 1)
        with pytest.raises(fca.FcaError) as err:
            ctx.enumerate(capacity=want.shape[0])
        assert err.value.status == fca.FCA_ERR_CUDA
        assert "waited past its limit" in str(err.value)
        ctx.set_option(fca.FCA_OPT_WAIT_LIMIT_NS, 0)
        got = ctx.enumerate(capacity=want.shape[0]).cpu().numpy().view(np.uint32)
        assert same_set(got, want)


# Small planted-block tables (the planted-bicluster recipe at other sizes): many extents of 65 to a
# few hundred objects, which are stored as object-id lists and expanded one per warp by the mid-tier
# kernel, beside larger ones for the bitmap-tier kernel.
LIST_TIER_CASES = [(4000, 48, 0.03, 6, (80, 400), (4, 10), 1), (5000, 64, 0.05, 10, (100, 600), (4, 12), 3),
                   (8000, 100, 0.03, 14, (150, 900), (5, 12), 6), (40000, 33, 0.02, 8, (100, 3000), (3, 8), 5)]


@pytest.mark.parametrize("mode", ["mid_kernel", "mid_kernel_no_inherit", "default", "mid_off", "lists_off"])
@pytest.mark.parametrize("case", LIST_TIER_CASES)
def test_list_tier_modes(case, mode, monkeypatch):
    """The same intents and closures whichever kernel takes the extents of 65 to a few hundred
    objects: the mid-tier kernel on every mid level (FCA_MID_MIN=1), with and without the failures
    its entries inherit from their mid-tier ancestors (FCA_NO_INHERIT=1: every candidate's closure
    is computed), the default choice (these levels are small, so the block-wide kernel takes the mid
    pools), the bitmap-tier kernel reading id lists from the big pools (FCA_MID_MAX=0), or the
    bitmap-tier kernel on N-bit bitmaps only (FCA_LIST_MAX=0). The closure count includes the
    candidates skipped by inheritance, so it matches the oracle's in every mode."""
    n, m, p, blocks, objects, attrs, seed = case
    if mode.startswith("mid_kernel"):
        monkeypatch.setenv("FCA_MID_MIN", "1")
    if mode == "mid_kernel_no_inherit":
        monkeypatch.setenv("FCA_NO_INHERIT", "1")
    elif mode == "mid_off":
        monkeypatch.setenv("FCA_MID_MAX", "0")
    elif mode == "lists_off":
        monkeypatch.setenv("FCA_LIST_MAX", "0")
    rows = cx.planted_context(n, m, p, blocks, objects, attrs, seed)
    _, st = check_against_oracle(rows, n, m, threads=8)
    if mode.startswith("mid_kernel"):
        assert st["mid_launches"] > 0
    elif mode != "default":
        assert st["mid_launches"] == 0
    if mode in ("mid_kernel", "mid_kernel_no_inherit", "default", "mid_off"):
        assert st["list_max"] > 64
    if mode in ("mid_kernel", "mid_kernel_no_inherit", "default"):
        assert st["mid_max"] == min(256, st["list_max"])


@pytest.mark.parametrize("m", [128, 256, 96])
def test_output_buffer_alignment(m):
    """The output rows are mapped back to attribute order in place, with 16-byte vector accesses when
    the rows are a multiple of four words and the caller's buffer is 16-byte aligned, word by word
    otherwise: a buffer that starts 4 bytes past an aligned address must give the same rows, and
    the word before it must stay untouched."""
    import torch
    from closed_set_enumeration_gb300 import fca
    n = 3000
    rows = cx.random_context(n, m, 0.04, 7)
    ref = oracle.cbo(rows, n, m, threads=8)["intents"]
    wm = (m + 31) // 32
    k = ref.shape[0]
    for offset in (0, 1):
        buf = torch.full((k * wm + offset + 1,), -7, dtype=torch.int32, device="cuda")
        out = buf[offset:offset + k * wm].view(k, wm)
        with fca.Context(rows, n, m) as ctx:
            st, cnt = ctx.enumerate_into(out, k)
        assert st == fca.FCA_OK and cnt == k
        got = out.cpu().numpy().view(np.uint32)
        assert same_set(got, ref)
        host = buf.cpu().numpy()
        if offset:
            assert host[0] == -7
        assert host[-1] == -7


@pytest.mark.parametrize("mid_min", [None, "1"])
def test_inherited_failures_past_the_child_lists(mid_min, monkeypatch):
    """A mid-tier node with more level children than a node records for its inherited failures
    (32 per mid node, 64 per bitmap-tier work item): the 200 objects holding attribute 0 form a node
    of the mid tier (9 000 objects, so id lists reach 256) whose 36 candidates are held by 80 of them
    each, so most of its children are mid-tier nodes again. Those past the recorded ones inherit no
    failures; the intents and the closure count must still be the oracle's, with the mid kernel on
    every mid level (FCA_MID_MIN=1) and with the default choice."""
    if mid_min:
        monkeypatch.setenv("FCA_MID_MIN", mid_min)
    rng = np.random.default_rng(11)
    n, m = 9000, 64
    cells = np.zeros((n, m), dtype=bool)
    cells[:200, 0] = True
    for a in range(1, 37):
        cells[rng.choice(200, 80, replace=False), a] = True
    cells[200:, 50:] = rng.random((n - 200, 14)) < 0.1
    rows = cx.pack_rows(cells)
    _, st = check_against_oracle(rows, n, m, threads=8)
    assert st["mid_max"] == 256
    if mid_min:
        assert st["mid_launches"] > 0


def test_growth_ahead_of_launches():
    """With tiny initial pools, the first call grows each level's destinations ahead of its launch
    from the previous launch's children per parent: fewer launches are rolled back than without it
    (FCA_PREGROW=0), and the intents and closures are the oracle's either way."""
    n, m = 4000, 60
    rows = cx.random_context(n, m, 0.12, 12)
    rows[: n // 4, 0] |= np.uint32(0x00FF00FF)
    ref = oracle.cbo(rows, n, m, threads=8)
    retries = {}
    for mode in ("1", "0"):
        mp = pytest.MonkeyPatch()
        mp.setenv("FCA_LEVEL_BYTES", "1")
        mp.setenv("FCA_QUEUE_ENTRIES", "1")
        mp.setenv("FCA_PREGROW", mode)
        try:
            got, st = gpu_run(rows, n, m, capacity=ref["intents"].shape[0] + 1)
        finally:
            mp.undo()
        assert not has_duplicates(got)
        assert same_set(got, ref["intents"])
        assert st["closures"] == ordered_closures(rows, n, m, threads=8)
        retries[mode] = st["retries"]
    assert retries["1"] < retries["0"]
