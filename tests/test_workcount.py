"""Pins of the work-counting pass (oracle/workcount.c) that gives the roofline its numerator.

Each count is defined per unit of the Close-by-One search (FCbO-to-CUDA page, sections 2.1-2.3,
3.1, 4.2): per parent its extent words, per candidate the words of the extent intersection and of
the cheaper closure route (rows or columns), per canonical child its frontier entry and output row.
The pins: a case worked by hand, a second implementation written here from the same definitions
(plain Python integers as bitsets), the relation to the oracle's own counts, and invariance to the
number of threads.
"""
import numpy as np
import pytest

import oracle
from oracle.workcount import workcount, derived
from closed_set_enumeration_gb300 import contexts as cx


def _words(bits: int, nwords: int):
    return [(bits >> (32 * w)) & 0xFFFFFFFF for w in range(nwords)]


def python_workcount(rows: np.ndarray, n: int, m: int, routes=None):
    """The counting definitions restated with Python integers (one bit per object / attribute).

    ``routes``, when a dict, also receives the totals of each closure route on its own.
    """
    wn, wm = (n + 31) // 32, (m + 31) // 32
    mask_m = (1 << m) - 1
    row = [int(sum(int(rows[o, w]) << (32 * w) for w in range(rows.shape[1]))) & mask_m for o in range(n)]
    col = [sum(1 << o for o in range(n) if (row[o] >> a) & 1) for a in range(m)]
    tiers = {t: dict(parents=0, closures=0, children=0, isect_words=0, closure_words=0, canon_words=0,
                     hbm_words=0) for t in ("list", "bitmap")}

    def intent(ext):
        d = mask_m
        for o in range(n):
            if (ext >> o) & 1:
                d &= row[o]
        return d

    def visit(a, b, y):
        t = tiers["bitmap" if bin(a).count("1") > 64 else "list"]
        t["parents"] += 1
        t["hbm_words"] += wn
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
            visit(c, d, j + 1)

    top = (1 << n) - 1
    visit(top, intent(top), 0)
    return tiers


def test_hand_worked_two_objects():
    # objects: o0 = {a0}, o1 = {a1}. Concepts: top (G, {}), ({o0}, {a0}), ({o1}, {a1}), ({}, M).
    # Parents 4 (every concept), closures 3 (top: j=0, j=1; {o0}: j=1), children 3.
    # Intersections: one word each (3). Closure words: top j=0 -> C={o0}, rows 1, columns: k=1
    # probes one word (violated) -> 1; top j=1 -> 1; {o0} j=1 -> C empty, rows route 0 -> 0.
    # HBM: 4 parent extents x 1 word + 3 children x (1 + 1 + 1) = 13.
    rows = np.array([[0b01], [0b10]], dtype=np.uint32)
    got = workcount(rows, 2, 2)
    assert got["list"] == dict(parents=4, closures=3, children=3, isect_words=3, closure_words=2,
                               canon_words=3, hbm_words=13)
    assert all(v == 0 for v in got["bitmap"].values())


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
    parents = got["list"]["parents"] + got["bitmap"]["parents"]
    closures = got["list"]["closures"] + got["bitmap"]["closures"]
    children = got["list"]["children"] + got["bitmap"]["children"]
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
