"""Pins of the work-counting pass (oracle/workcount.c) that gives the roofline its numerator.

Each count is defined per unit of the Close-by-One search (FCbO-to-CUDA page, sections 2.1-2.3,
3.1, 4.2): per parent its extent words, per candidate the words of the extent intersection and of
the cheaper closure route (rows or columns), per canonical child its frontier entry and output row.
The pins: a case worked by hand, a second implementation written here from the same definitions
(plain Python integers as bitsets), the relation to the oracle's own counts, invariance to the
number of threads, and the split of the tiers by extent size (object-list tier up to 64 objects,
mid tier up to a threshold, bitmap tier above it), which moves counts between tiers without
changing their sums.
"""
import numpy as np
import pytest

import oracle
from oracle.workcount import workcount, derived
from closed_set_enumeration_gb300 import contexts as cx


def _words(bits: int, nwords: int):
    return [(bits >> (32 * w)) & 0xFFFFFFFF for w in range(nwords)]


def python_workcount(rows: np.ndarray, n: int, m: int, routes=None, mid_max: int = 0, list_max: int = 0):
    """The counting definitions restated with Python integers (one bit per object / attribute).

    ``routes``, when a dict, also receives the totals of each closure route on its own. The lean
    model's words follow the tiered representation: an id list per extent of at most 64 objects or
    at most ``list_max`` objects (else a bitmap of W_N words), object-list subtrees searched in
    place (only their roots are read), rows gathered once per parent kept as an id list.
    """
    wn, wm = (n + 31) // 32, (m + 31) // 32
    mask_m = (1 << m) - 1
    row = [int(sum(int(rows[o, w]) << (32 * w) for w in range(rows.shape[1]))) & mask_m for o in range(n)]
    col = [sum(1 << o for o in range(n) if (row[o] >> a) & 1) for a in range(m)]
    tiers = {t: dict(parents=0, closures=0, children=0, isect_words=0, closure_words=0, canon_words=0,
                     hbm_words=0, hbm_lean_words=0, l2_lean_words=0) for t in ("list", "mid", "bitmap")}

    def tier_name(size):
        return "list" if size <= 64 else ("mid" if size <= mid_max else "bitmap")

    def entry(size):
        return size if size <= 64 or size <= list_max else wn

    def intent(ext):
        d = mask_m
        for o in range(n):
            if (ext >> o) & 1:
                d &= row[o]
        return d

    def visit(a, b, y, up):
        size = bin(a).count("1")
        tn = tier_name(size)
        t = tiers[tn]
        t["parents"] += 1
        t["hbm_words"] += wn
        as_list = tn != "bitmap" or size <= list_max
        if not (tn == "list" and up == "list"):
            t["hbm_lean_words"] += entry(size)
            if as_list:
                t["l2_lean_words"] += size * wm
        a_words = [w for w, v in enumerate(_words(a, wn)) if v]
        for j in range(y, m):
            if (b >> j) & 1:
                continue
            t["closures"] += 1
            t["isect_words"] += len(a_words)
            c = a & col[j]
            cw = [(w, v) for w, v in enumerate(_words(c, wn)) if v]
            rows_route = bin(c).count("1") * wm
            total = 0
            for k in range(m):
                if k == j or (b >> k) & 1:
                    continue
                ck = _words(col[k], wn)
                probed, inside = 0, True
                for w, v in cw:
                    probed += 1
                    if v & ~ck[w] & 0xFFFFFFFF:
                        inside = False
                        break
                total += probed
                if inside and k < j:
                    break
            t["closure_words"] += min(total, rows_route)
            if not as_list:
                t["l2_lean_words"] += len(a_words) + min(total, rows_route)
            if routes is not None:
                routes["rows"] = routes.get("rows", 0) + rows_route
                routes["columns"] = routes.get("columns", 0) + total
            t["canon_words"] += wm
            d = intent(c)
            below = (1 << j) - 1
            if (d ^ b) & below:
                continue
            t["children"] += 1
            t["hbm_words"] += wn + 2 * wm
            csize = bin(c).count("1")
            t["hbm_lean_words"] += wm
            if not (tn == "list" and tier_name(csize) == "list"):
                t["hbm_lean_words"] += entry(csize) + wm
            visit(c, d, j + 1, tn)

    top = (1 << n) - 1
    visit(top, intent(top), 0, None)
    return tiers


def test_hand_worked_two_objects():
    # objects: o0 = {a0}, o1 = {a1}. Concepts: top (G, {}), ({o0}, {a0}), ({o1}, {a1}), ({}, M).
    # Parents 4 (every concept), closures 3 (top: j=0, j=1; {o0}: j=1), children 3.
    # Intersections: one word each (3). Closure words: top j=0 -> C={o0}, rows 1, columns: k=1
    # probes one word (violated) -> 1; top j=1 -> 1; {o0} j=1 -> C empty, rows route 0 -> 0.
    # HBM: 4 parent extents x 1 word + 3 children x (1 + 1 + 1) = 13.
    # Lean model: the top is the only object-list root: its 2 ids and 2 x 1 row words; every other
    # node lives in the searching warp; each child writes its output row (3 x 1 word).
    rows = np.array([[0b01], [0b10]], dtype=np.uint32)
    got = workcount(rows, 2, 2)
    assert got["list"] == dict(parents=4, closures=3, children=3, isect_words=3, closure_words=2,
                               canon_words=3, hbm_words=13, hbm_lean_words=5, l2_lean_words=2)
    assert all(v == 0 for v in got["bitmap"].values())
    assert all(v == 0 for v in got["mid"].values())


@pytest.mark.parametrize("n,m,p,seed", [(5, 4, 0.5, 0), (12, 7, 0.4, 1), (30, 9, 0.3, 2), (40, 10, 0.5, 3),
                                        (70, 8, 0.6, 4), (90, 6, 0.7, 5)])
def test_matches_python_restatement(n, m, p, seed):
    rows = cx.random_context(n, m, p, seed)
    assert workcount(rows, n, m) == python_workcount(rows, n, m)


@pytest.mark.parametrize("name", ["tiny"])
def test_relations_to_the_oracle(name):
    w = cx.WORKLOADS[name]
    rows = w.rows()
    got = workcount(rows, w.n_objects, w.n_attrs)
    ref = oracle.cbo(rows, w.n_objects, w.n_attrs)
    concepts = ref["intents"].shape[0]
    parents = sum(t["parents"] for t in got.values())
    closures = sum(t["closures"] for t in got.values())
    children = sum(t["children"] for t in got.values())
    assert parents == concepts            # every concept is expanded once
    assert children == concepts - 1       # every concept but the top is some node's child
    assert closures == ref["closures"]
    for t in got.values():
        assert t["canon_words"] == t["closures"] * ((w.n_attrs + 31) // 32)
        d = derived(t)
        assert d["ops"] >= d["l2_words"] >= t["isect_words"]


def test_thread_split_does_not_change_counts():
    rows = cx.random_context(300, 24, 0.25, 7)
    one = workcount(rows, 300, 24, threads=1)
    assert workcount(rows, 300, 24, threads=5) == one
    assert one["bitmap"]["parents"] > 0 and one["list"]["parents"] > 0


def test_closure_route_takes_the_cheaper_one():
    # On this context neither route alone gives the counted total: a count that took only the
    # rows or only the columns would fail here.
    rows = cx.random_context(200, 12, 0.5, 11)
    routes = {}
    ref = python_workcount(rows, 200, 12, routes)
    got = workcount(rows, 200, 12)
    assert got == ref
    total_close = sum(t["closure_words"] for t in got.values())
    assert 0 < total_close < routes["rows"]
    assert total_close < routes["columns"]


@pytest.mark.parametrize("mid_max", [64, 80, 120, 1000])
def test_mid_tier_split(mid_max):
    """Parents of 65..mid_max objects are counted in the mid tier: the C pass and the Python
    restatement agree, the mid tier is empty at 64 and takes the whole large tier at N, and every
    count of mid + bitmap equals the bitmap tier of the two-tier split (the lean model's too, with
    every large extent kept as an id list in both)."""
    rows = cx.random_context(160, 9, 0.55, 12)
    got = workcount(rows, 160, 9, mid_max=mid_max, list_max=1000)
    assert got == python_workcount(rows, 160, 9, mid_max=mid_max, list_max=1000)
    two = workcount(rows, 160, 9, list_max=1000)
    assert got["list"] == two["list"]
    for f in two["bitmap"]:
        assert got["mid"][f] + got["bitmap"][f] == two["bitmap"][f]
    if mid_max == 64:
        assert all(v == 0 for v in got["mid"].values())
    if mid_max >= 160:
        assert all(v == 0 for v in got["bitmap"].values())
    if mid_max in (80, 120):
        assert got["mid"]["parents"] > 0 and got["bitmap"]["parents"] > 0


def test_stored_counts_are_reproduced():
    """The stored counts of the smaller workloads (tests/golden/work_counts.json) are what the
    counting pass gives now, in the stored processing order and tier split."""
    import json
    import os
    from tests._util import GOLDEN, support_order
    table = json.load(open(os.path.join(GOLDEN, "work_counts.json")))
    for name in ("tiny", "sparse"):
        entry = table[name]
        w = cx.WORKLOADS[name]
        rows = w.rows()
        if entry.get("order") == "support":
            rows = support_order(rows, w.n_objects, w.n_attrs)[0]
        got = workcount(rows, w.n_objects, w.n_attrs, threads=4, mid_max=entry.get("mid_max", 0),
                        list_max=entry.get("list_max", 0))
        for tier, counts in entry["tiers"].items():
            assert got[tier] == counts, (name, tier)


@pytest.mark.parametrize("list_max", [0, 70, 100, 1000])
def test_lean_model(list_max):
    """The lean model against its restatement and its extremes: with every extent an id list the
    large tiers gather rows and read ids only; with none (list_max 0) a large parent reads W_N
    words and its candidates' L2 words equal the bitmap model's intersection and closure words.
    Object-list subtrees read their roots only, and their children other than new roots write
    their output rows only."""
    n, m = 300, 12
    rows = cx.random_context(n, m, 0.5, 13)
    got = workcount(rows, n, m, threads=3, list_max=list_max)
    assert got == python_workcount(rows, n, m, list_max=list_max)
    big = got["bitmap"]
    if list_max == 0:
        assert big["l2_lean_words"] == big["isect_words"] + big["closure_words"]
    assert got["list"]["hbm_lean_words"] < got["list"]["hbm_words"]
    assert got["list"]["hbm_lean_words"] >= got["list"]["children"] * ((m + 31) // 32)


# ---- lower-cover search (oracle/coverwork.c)

def python_coverwork(rows: np.ndarray, n: int, m: int, intents: np.ndarray):
    """The cover-search counts restated from their definitions, with plain Python integers as
    bitsets: per concept (A, B), W_N extent words, (M - |B|) * nnzw(A) intersection words, and
    |C_k| * W_M closure words for every k outside B with C_k = A & column k non-empty."""
    wn, wm = (n + 31) // 32, (m + 31) // 32
    row_bits = []
    for o in range(n):
        v = 0
        for w in range(wm):
            v |= int(rows[o, w]) << (32 * w)
        row_bits.append(v & ((1 << m) - 1))
    out = {"concepts": 0, "extent_words": 0, "isect_words": 0, "closure_words": 0}
    for r in range(intents.shape[0]):
        b = 0
        for w in range(wm):
            b |= int(intents[r, w]) << (32 * w)
        ext = [o for o in range(n) if row_bits[o] & b == b]
        nnzw = len({o // 32 for o in ext})
        out["concepts"] += 1
        out["extent_words"] += wn
        out["isect_words"] += (m - bin(b).count("1")) * nnzw
        for k in range(m):
            if (b >> k) & 1:
                continue
            ck = sum(1 for o in ext if (row_bits[o] >> k) & 1)
            out["closure_words"] += ck * wm
    return out


def test_coverwork_hand_worked():
    """Two objects with one attribute each: concepts {} (both objects), {a0}, {a1}, {a0, a1} (no
    object). Intersections: 2 + 1 + 1 + 0 words; closures: the two singletons under {} only."""
    from oracle.workcount import coverwork
    rows = np.array([[0b01], [0b10]], dtype=np.uint32)
    intents = np.array([[0b00], [0b01], [0b10], [0b11]], dtype=np.uint32)
    assert coverwork(rows, 2, 2, intents) == {"concepts": 4, "extent_words": 4, "isect_words": 4,
                                               "closure_words": 2}


@pytest.mark.parametrize("n,m,p,seed", [(40, 12, 0.3, 1), (70, 33, 0.2, 2), (100, 40, 0.15, 3)])
def test_coverwork_matches_python_restatement(n, m, p, seed):
    """The C count against the Python restatement on the oracle's full intent set, across word
    boundaries of N and M, and independent of the thread split and of the order of the intents."""
    from oracle.workcount import coverwork
    rows = cx.random_context(n, m, p, seed)
    intents = oracle.cbo(rows, n, m)["intents"]
    want = python_coverwork(rows, n, m, intents)
    assert coverwork(rows, n, m, intents, threads=1) == want
    assert coverwork(rows, n, m, intents[::-1].copy(), threads=3) == want
