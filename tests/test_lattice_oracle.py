"""Pins for the lattice oracle (extents of intents, cover edges): checked against closed forms of
textbook contexts and against a pure-Python set enumeration on tiny contexts, never against itself.

- contranominal scale (object i lacks only attribute i): every attribute set is an intent, the
  extent of B is the objects outside B, and the lattice is the Boolean lattice: n * 2^(n-1) cover
  edges, each adding exactly one attribute;
- chain (object i has attributes 0..i): the intents are the n prefixes, the extent of the prefix
  0..i is the objects i..n-1, and the lattice is a chain of n - 1 edges;
- identity (object i has only attribute i): top, the n singletons and the bottom; 2n edges;
- Hasse-diagram invariants: only the top lacks an upper cover, only the bottom a lower cover, and
  every edge goes from an intent to a proper superset;
- pure-Python brute force on tiny random contexts (intents as frozensets, the cover relation by
  three nested loops);
- planted mistakes in a copy of the cover oracle each fail one of the above;
- the rule the cover kernel computes (lower covers = the maximal distinct restrictions A & {k}',
  each with intent B plus the attributes giving the same set), restated with Python sets, equals
  the oracle's cover relation; and the oracle's two formulations (whole relation, one concept's
  lower covers) agree on a thousand-concept lattice;
- the facts behind the cover kernel's shortcuts hold in the oracle's relation: an empty restriction
  is a cover's extent only when all restrictions are empty (the one cover is then the concept with
  the empty extent), and the attributes holding a non-empty restriction are those its objects share.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import lattice
from closed_set_enumeration_gb300 import contexts as cx
from tests._util import attrs_to_row


def intent_sets(intents, m):
    cells = cx.unpack_rows(np.ascontiguousarray(intents, dtype=np.uint32), m)
    return [frozenset(np.nonzero(c)[0].tolist()) for c in cells]


def chain(n):
    """Object i has attributes 0..i (n x n)."""
    return cx.pack_rows(np.tril(np.ones((n, n), dtype=bool)))


# ---------------------------------------------------------------- extents

@pytest.mark.parametrize("n", [1, 4, 9, 33])
def test_extent_contranominal_is_complement(n):
    rows = cx.contranominal(n)
    rng = np.random.default_rng(n)
    for _ in range(20):
        b = set(np.nonzero(rng.random(n) < 0.4)[0].tolist())
        ext = oracle.derive_extent(rows, attrs_to_row(sorted(b), n))
        assert set(np.nonzero(ext)[0].tolist()) == set(range(n)) - b


@pytest.mark.parametrize("n", [3, 32, 40])
def test_extent_chain_is_suffix(n):
    rows = chain(n)
    for i in range(n):
        ext = oracle.derive_extent(rows, attrs_to_row(range(i + 1), n))
        assert np.nonzero(ext)[0].tolist() == list(range(i, n))
    # the empty set: every object; a non-prefix set {i}: objects i..n-1 as well
    assert oracle.derive_extent(rows, attrs_to_row([], n)).all()


def test_extent_matches_cell_loops():
    n, m = 13, 37
    rows = cx.random_context(n, m, 0.6, 3)
    cells = cx.unpack_rows(rows, m)
    rng = np.random.default_rng(4)
    for _ in range(40):
        b = [a for a in range(m) if rng.random() < 0.1]
        want = [o for o in range(n) if all(cells[o][a] for a in b)]
        got = np.nonzero(oracle.derive_extent(rows, attrs_to_row(b, m)))[0].tolist()
        assert got == want


# ---------------------------------------------------------------- cover edges: closed forms

@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_covers_boolean_lattice(n):
    rows = cx.contranominal(n)
    intents = oracle.cbo(rows, n, n)["intents"]
    e = lattice.cover_edges(intents, n)
    assert e.shape[0] == n * 2 ** (n - 1)
    sets = intent_sets(intents, n)
    for i, j in e:
        assert sets[i] < sets[j] and len(sets[j]) == len(sets[i]) + 1


@pytest.mark.parametrize("n", [1, 2, 5, 33])
def test_covers_chain(n):
    rows = chain(n)
    intents = oracle.cbo(rows, n, n)["intents"]
    assert intents.shape[0] == n
    sets = intent_sets(intents, n)
    e = lattice.cover_edges(intents, n)
    assert e.shape[0] == n - 1
    for i, j in e:
        assert sets[i] == frozenset(range(len(sets[i]))) and len(sets[j]) == len(sets[i]) + 1


@pytest.mark.parametrize("n", [2, 3, 7, 40])
def test_covers_identity(n):
    rows = cx.identity(n)
    intents = oracle.cbo(rows, n, n)["intents"]
    sets = intent_sets(intents, n)
    e = lattice.cover_edges(intents, n)
    assert e.shape[0] == 2 * n
    for i, j in e:
        assert (len(sets[i]), len(sets[j])) in ((0, 1), (1, n))


# ---------------------------------------------------------------- invariants and brute force

def brute_covers(sets):
    """Cover pairs by three nested loops over Python frozensets."""
    out = []
    for i, a in enumerate(sets):
        for j, b in enumerate(sets):
            if a < b and not any(a < c < b for c in sets):
                out.append((i, j))
    return sorted(out)


@pytest.mark.parametrize("n,m,p,seed", [(6, 5, 0.5, 1), (9, 8, 0.4, 2), (12, 10, 0.45, 3), (7, 35, 0.7, 4)])
def test_covers_match_brute_force(n, m, p, seed):
    rows = cx.random_context(n, m, p, seed)
    intents = oracle.cbo(rows, n, m)["intents"]
    sets = intent_sets(intents, m)
    e = lattice.cover_edges(intents, m)
    assert sorted(map(tuple, e.tolist())) == brute_covers(sets)
    for i in range(len(sets)):
        want = [j for (a, j) in brute_covers(sets) if a == i]
        assert lattice.lower_covers_of(intents, m, i).tolist() == want


@pytest.mark.parametrize("n,m,p,seed", [(60, 12, 0.35, 5), (100, 20, 0.2, 6)])
def test_hasse_invariants(n, m, p, seed):
    rows = cx.random_context(n, m, p, seed)
    intents = oracle.cbo(rows, n, m)["intents"]
    k = intents.shape[0]
    e = lattice.cover_edges(intents, m)
    has_up = np.zeros(k, bool)
    has_down = np.zeros(k, bool)
    has_up[e[:, 1]] = True
    has_down[e[:, 0]] = True
    sizes = np.array([len(s) for s in intent_sets(intents, m)])
    top, bottom = int(np.argmin(sizes)), int(np.argmax(sizes))
    assert not has_up[top] and has_up.sum() == k - 1
    assert not has_down[bottom] and has_down.sum() == k - 1
    assert np.all(sizes[e[:, 1]] > sizes[e[:, 0]])
    # the order is graded by nothing in general, but a path of covers exists from top to every node
    reach = {top}
    frontier = [top]
    adj = {}
    for i, j in e.tolist():
        adj.setdefault(i, []).append(j)
    while frontier:
        nxt = []
        for i in frontier:
            for j in adj.get(i, []):
                if j not in reach:
                    reach.add(j)
                    nxt.append(j)
        frontier = nxt
    assert len(reach) == k


# ---------------------------------------------------------------- planted mistakes

def _mutant_nonproper(intents, m):
    """Inclusion taken as 'subset or equal': self-loops appear."""
    cells = lattice._bits(intents, m).astype(np.float32)
    size = cells.sum(axis=1)
    outside = size[:, None] - cells @ cells.T
    proper = outside == 0
    p = proper.astype(np.float32)
    cover = proper & ~((p @ p) > 0)
    return np.argwhere(cover)


def _mutant_no_between(intents, m):
    """The 'nothing in between' condition dropped: every comparable pair is an edge."""
    cells = lattice._bits(intents, m).astype(np.float32)
    size = cells.sum(axis=1)
    outside = size[:, None] - cells @ cells.T
    return np.argwhere((outside == 0) & (size[None, :] > size[:, None]))


def _mutant_transposed(intents, m):
    """Edges written as (lower, upper)."""
    return lattice.cover_edges(intents, m)[:, ::-1]


@pytest.mark.parametrize("mutant", [_mutant_nonproper, _mutant_no_between, _mutant_transposed])
def test_planted_cover_mistakes_are_caught(mutant):
    caught = False
    for n in (3, 4):
        intents = oracle.cbo(cx.contranominal(n), n, n)["intents"]
        e = np.asarray(mutant(intents, n))
        sets = intent_sets(intents, n)
        ok = e.shape[0] == n * 2 ** (n - 1) and all(
            sets[i] < sets[j] and len(sets[j]) == len(sets[i]) + 1 for i, j in e)
        caught |= not ok
    assert caught


# ---------------------------------------------------------------- the rule the cover kernel uses

def covers_by_maximal_restrictions(rows, n, m, intents):
    """Lower covers of each concept (A, B) as the maximal distinct sets C_k = A & {k}' over k not in
    B, each with intent B + {k2 : C_k2 = C_k}, emitted once from its smallest k (plain Python sets)."""
    cells = cx.unpack_rows(rows, m)
    sets = intent_sets(intents, m)
    row_of = {s: i for i, s in enumerate(sets)}
    out = []
    for i, b in enumerate(sets):
        a = frozenset(o for o in range(n) if all(cells[o][x] for x in b))
        c = {k: frozenset(o for o in a if cells[o][k]) for k in range(m) if k not in b}
        for k, ck in c.items():
            dominated = any(ck < c2 for c2 in c.values())
            first = min(k2 for k2, c2 in c.items() if c2 == ck) == k
            if dominated or not first:
                continue
            d = b | {k2 for k2, c2 in c.items() if c2 == ck}
            out.append((i, row_of[frozenset(d)]))
    return sorted(out)


@pytest.mark.parametrize("n,m,p,seed", [(20, 8, 0.4, 1), (40, 12, 0.3, 2), (70, 40, 0.2, 3), (15, 6, 0.6, 4)])
def test_maximal_restrictions_give_the_covers(n, m, p, seed):
    rows = cx.random_context(n, m, p, seed)
    intents = oracle.cbo(rows, n, m)["intents"]
    assert covers_by_maximal_restrictions(rows, n, m, intents) == \
        sorted(map(tuple, lattice.cover_edges(intents, m).tolist()))


@pytest.mark.parametrize("n,m,p,seed", [(20, 8, 0.4, 1), (40, 12, 0.3, 2), (70, 40, 0.2, 3), (30, 10, 0.05, 5)])
def test_empty_restrictions_and_row_closures(n, m, p, seed):
    """The two facts the cover kernel's shortcuts rest on, against the oracle's cover relation. An
    empty C_k = A & {k}' is a lower cover's extent only when every C_k outside B is empty, and then
    the concept's one lower cover has the empty extent. The attributes k2 outside B whose C_k2 holds
    a non-empty C_k are exactly those common to all of C_k's objects."""
    rows = cx.random_context(n, m, p, seed)
    cells = cx.unpack_rows(rows, m)
    intents = oracle.cbo(rows, n, m)["intents"]
    sets = intent_sets(intents, m)
    lower = {}
    for i, j in lattice.cover_edges(intents, m).tolist():
        lower.setdefault(i, []).append(j)
    seen_all_empty = seen_some = 0
    for i, b in enumerate(sets):
        a = frozenset(o for o in range(n) if all(cells[o][x] for x in b))
        c = {k: frozenset(o for o in a if cells[o][k]) for k in range(m) if k not in b}
        cover_extents = [frozenset(o for o in range(n) if all(cells[o][x] for x in sets[j]))
                         for j in lower.get(i, [])]
        if c and all(not ck for ck in c.values()):
            seen_all_empty += 1
            assert cover_extents == [frozenset()]
        elif c:
            seen_some += 1
            assert frozenset() not in cover_extents
        for k, ck in c.items():
            if ck:
                common = {x for x in range(m) if all(cells[o][x] for o in ck)}
                assert common - b == {k2 for k2, c2 in c.items() if ck <= c2}
    assert seen_all_empty and seen_some


def test_two_cover_formulations_agree_at_a_thousand_concepts():
    rows = cx.random_context(1000, 30, 0.1, 11)
    intents = oracle.cbo(rows, 1000, 30)["intents"]
    e = lattice.cover_edges(intents, 30)
    by_row = {}
    for i, j in e.tolist():
        by_row.setdefault(i, []).append(j)
    rng = np.random.default_rng(2)
    for i in rng.choice(intents.shape[0], 120, replace=False):
        assert lattice.lower_covers_of(intents, 30, int(i)).tolist() == sorted(by_row.get(int(i), []))
