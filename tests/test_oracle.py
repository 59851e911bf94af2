"""Pins for the CPU oracle: it is checked against things other than itself.

- hand-derived golden fixtures (tests/golden/);
- closed forms of textbook contexts (contranominal scale: 2^n concepts, the
  FCbO-to-CUDA page's worst case 2^min(|G|,|M|) of section 1.3; identity:
  n + 2; all-zero: 2; all-ones: 1; one object: 2 or 1) and the exact
  closure / depth counts of the Close-by-One tree on them;
- brute force: closing every attribute subset (M <= 16) and deriving every
  object subset (N <= 16, any M, which pins the multi-word logic);
- invariants: fixed points B'' = B, no duplicates, top and bottom present,
  object- and attribute-permutation invariance, duality |K| = |K^T|, and
  closure of intents under intersection;
- mutation checks: plausible mistakes planted in a copy of the oracle source
  must each fail at least one of the pins above.
"""
import itertools
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from closed_set_enumeration_gb300 import contexts as cx
from tests._util import (golden_names, has_duplicates, load_golden, same_set, sort_rows,
                         attrs_to_row)


def full_row(m):
    return attrs_to_row(range(m), m)


# ---------------------------------------------------------------- golden

@pytest.mark.parametrize("name", golden_names())
def test_golden_oracle(name):
    n, m, rows, expected = load_golden(name)
    got = oracle.cbo(rows, n, m)["intents"]
    assert same_set(got, expected), name


@pytest.mark.parametrize("name", golden_names())
def test_golden_brute_force(name):
    n, m, rows, expected = load_golden(name)
    assert same_set(oracle.brute_force_by_objects(rows, n, m), expected)
    if m <= 16:
        assert same_set(oracle.brute_force(rows, n, m), expected)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 12, 16])
def test_contranominal_has_2_pow_n(n):
    rows = cx.contranominal(n)
    r = oracle.cbo(rows, n, n)
    assert r["intents"].shape[0] == 2 ** n
    assert not has_duplicates(r["intents"])
    # every subset is closed, so every candidate is canonical: one closure per child
    assert r["closures"] == 2 ** n - 1
    # depth d holds the d-element subsets
    from math import comb
    assert [int(x) for x in r["depth_counts"][: n + 1]] == [comb(n, d) for d in range(n + 1)]
    if n <= 12:
        assert oracle.brute_force(rows, n, n).shape[0] == 2 ** n


@pytest.mark.parametrize("n", [2, 3, 7, 31, 32, 33, 64, 65, 100])
def test_identity_has_n_plus_2(n):
    rows = cx.identity(n)
    r = oracle.cbo(rows, n, n)
    assert r["intents"].shape[0] == n + 2
    # root: n candidates; singleton {j}: n-1-j candidates (all empty extents)
    assert r["closures"] == n + n * (n - 1) // 2
    expected = [attrs_to_row([], n), full_row(n)] + [attrs_to_row([j], n) for j in range(n)]
    assert same_set(r["intents"], np.stack(expected))


@pytest.mark.parametrize("n,m", [(1, 1), (3, 5), (40, 33), (70, 64), (5, 100)])
def test_all_zero_context(n, m):
    rows = np.zeros((n, (m + 31) // 32), dtype=np.uint32)
    r = oracle.cbo(rows, n, m)
    assert same_set(r["intents"], np.stack([attrs_to_row([], m), full_row(m)]))
    assert r["closures"] == m          # every top-level candidate has an empty extent


@pytest.mark.parametrize("n,m", [(1, 1), (4, 7), (33, 32), (2, 65)])
def test_all_ones_context(n, m):
    rows = np.tile(full_row(m), (n, 1))
    r = oracle.cbo(rows, n, m)
    assert same_set(r["intents"], full_row(m)[None, :])
    assert r["closures"] == 0


@pytest.mark.parametrize("m,attrs", [(5, [1, 3]), (40, [0, 31, 32, 39]), (64, []), (3, [0, 1, 2])])
def test_single_object(m, attrs):
    row = attrs_to_row(attrs, m)[None, :]
    r = oracle.cbo(row, 1, m)
    expect = {tuple(attrs_to_row(attrs, m)), tuple(full_row(m))}
    assert set(map(tuple, r["intents"])) == expect
    assert r["intents"].shape[0] == len(expect)


def test_padding_bits_ignored():
    m = 5
    rows = cx.random_context(20, m, 0.4, 7)
    dirty = rows | np.uint32(0xFFFFFFE0)
    a = oracle.cbo(rows, 20, m)["intents"]
    b = oracle.cbo(dirty, 20, m)["intents"]
    assert same_set(a, b)
    assert not np.any(b & np.uint32(0xFFFFFFE0))


# ---------------------------------------------------------------- brute force

RANDOM_TINY = [(n, m, d, s) for (n, m) in [(1, 4), (5, 5), (31, 9), (32, 12), (33, 16), (64, 16)]
               for d in (0.1, 0.3, 0.6) for s in (0, 1)]


@pytest.mark.parametrize("n,m,density,seed", RANDOM_TINY)
def test_oracle_matches_attribute_brute_force(n, m, density, seed):
    rows = cx.random_context(n, m, density, seed)
    got = oracle.cbo(rows, n, m)["intents"]
    assert not has_duplicates(got)
    assert same_set(got, oracle.brute_force(rows, n, m))


def test_tiny_workload_matches_brute_force():
    w = cx.WORKLOADS["tiny"]
    rows = w.rows()
    got = oracle.cbo(rows, w.n_objects, w.n_attrs)["intents"]
    assert same_set(got, oracle.brute_force(rows, w.n_objects, w.n_attrs))


@pytest.mark.parametrize("n,m,density,seed", [(5, 31, 0.5, 0), (12, 32, 0.5, 1), (16, 33, 0.6, 2),
                                              (16, 63, 0.5, 3), (16, 64, 0.7, 4), (14, 65, 0.6, 5),
                                              (16, 100, 0.6, 6), (16, 130, 0.8, 7), (9, 200, 0.9, 8)])
def test_oracle_matches_object_brute_force(n, m, density, seed):
    rows = cx.random_context(n, m, density, seed)
    got = oracle.cbo(rows, n, m)["intents"]
    assert not has_duplicates(got)
    assert same_set(got, oracle.brute_force_by_objects(rows, n, m))


def test_brute_forces_agree():
    for seed in range(4):
        rows = cx.random_context(12, 14, 0.45, seed)
        assert same_set(oracle.brute_force(rows, 12, 14), oracle.brute_force_by_objects(rows, 12, 14))


# ---------------------------------------------------------------- invariants

@pytest.fixture(scope="module")
def sparse_case():
    w = cx.WORKLOADS["sparse"]
    rows = w.rows()
    r = oracle.cbo(rows, w.n_objects, w.n_attrs, threads=4)
    return w, rows, r


def test_invariant_fixed_points(sparse_case):
    w, rows, r = sparse_case
    intents = r["intents"]
    rng = np.random.default_rng(11)
    pick = rng.choice(intents.shape[0], 1500, replace=False)
    for i in pick:
        b = intents[i]
        ext = oracle.derive_extent(rows, b)
        assert np.array_equal(oracle.derive_intent(rows, ext, w.n_attrs), b)


def test_invariant_no_duplicates_top_bottom(sparse_case):
    w, rows, r = sparse_case
    intents = r["intents"]
    assert not has_duplicates(intents)
    top = oracle.derive_intent(rows, np.ones(w.n_objects, bool), w.n_attrs)
    assert np.array_equal(intents[0], top)          # the top is output first
    s = set(map(tuple, intents))
    assert tuple(full_row(w.n_attrs)) in s


def test_invariant_intersection_closed(sparse_case):
    w, rows, r = sparse_case
    intents = r["intents"]
    s = set(map(tuple, intents))
    rng = np.random.default_rng(5)
    for _ in range(3000):
        i, j = rng.integers(0, intents.shape[0], 2)
        assert tuple(intents[i] & intents[j]) in s


def test_invariant_object_permutation(sparse_case):
    w, rows, r = sparse_case
    perm = np.random.default_rng(3).permutation(w.n_objects)
    r2 = oracle.cbo(rows[perm], w.n_objects, w.n_attrs, threads=4)
    assert same_set(r["intents"], r2["intents"])


def test_invariant_attribute_permutation(sparse_case):
    w, rows, r = sparse_case
    m = w.n_attrs
    perm = np.random.default_rng(4).permutation(m)       # new attribute k = old perm[k]
    cells = cx.unpack_rows(rows, m)
    r2 = oracle.cbo(cx.pack_rows(cells[:, perm]), w.n_objects, m, threads=4)
    got = cx.unpack_rows(r2["intents"], m)
    back = np.zeros_like(got)
    back[:, perm] = got
    assert same_set(cx.pack_rows(back), r["intents"])


@pytest.mark.parametrize("n,m,density,seed", [(40, 25, 0.3, 0), (200, 18, 0.25, 1), (64, 64, 0.15, 2)])
def test_invariant_duality(n, m, density, seed):
    rows = cx.random_context(n, m, density, seed)
    cells = cx.unpack_rows(rows, m)
    a = oracle.cbo(rows, n, m)
    b = oracle.cbo(cx.pack_rows(cells.T), m, n)
    assert a["intents"].shape[0] == b["intents"].shape[0]


@pytest.mark.parametrize("name,threads", [("sparse", 3), ("sparse", 8), ("tiny", 5)])
def test_thread_modes_agree(name, threads):
    w = cx.WORKLOADS[name]
    rows = w.rows()
    a = oracle.cbo(rows, w.n_objects, w.n_attrs, threads=1)
    b = oracle.cbo(rows, w.n_objects, w.n_attrs, threads=threads)
    assert same_set(a["intents"], b["intents"])
    assert a["closures"] == b["closures"]
    assert np.array_equal(a["depth_counts"], b["depth_counts"])


@pytest.mark.parametrize("n,m,density,seed,threads", [(300, 33, 0.2, 1, 1), (500, 64, 0.15, 2, 4),
                                                      (200, 100, 0.1, 3, 3)])
def test_digest_mode_matches_full_output(n, m, density, seed, threads):
    from tests._util import multiset_digest
    rows = cx.random_context(n, m, density, seed)
    full = oracle.cbo(rows, n, m, threads=threads)
    dig = oracle.cbo_digest(rows, n, m, threads=threads)
    assert dig["count"] == full["intents"].shape[0]
    assert dig["closures"] == full["closures"]
    assert np.array_equal(dig["depth_counts"], full["depth_counts"])
    assert (dig["hsum"], dig["hxor"]) == multiset_digest(full["intents"])
    # the digest tells sets apart: drop one intent, or change one bit of one
    assert multiset_digest(full["intents"][1:]) != (dig["hsum"], dig["hxor"])
    changed = full["intents"].copy()
    changed[3, 0] ^= np.uint32(1)
    assert multiset_digest(changed) != (dig["hsum"], dig["hxor"])


@pytest.mark.parametrize("n,m,density,seed,threads", [(300, 33, 0.2, 4, 2), (400, 70, 0.12, 5, 4),
                                                      (120, 16, 0.35, 6, 1)])
def test_relabeled_digest_is_the_original_tables_digest(n, m, density, seed, threads):
    """The intent set does not depend on how the attributes are numbered: searching the table with
    its columns in another order and renumbering each intent back must digest to the original
    table's full output. The permuted search evaluates other candidates (its closures differ from
    the original search's on these tables), so equal digests are not an artefact of equal work."""
    from tests._util import multiset_digest
    rows = cx.random_context(n, m, density, seed)
    full = oracle.cbo(rows, n, m, threads=threads)
    want = multiset_digest(full["intents"])
    perm = np.random.default_rng(seed).permutation(m)        # position r holds attribute perm[r]
    cells = cx.unpack_rows(rows, m)[:, perm]
    prows = cx.pack_rows(cells)
    got = oracle.cbo_digest(prows, n, m, threads=threads, label=perm)
    assert got["count"] == full["intents"].shape[0]
    assert (got["hsum"], got["hxor"]) == want
    assert got["closures"] == oracle.cbo(prows, n, m)["closures"]
    assert got["closures"] != full["closures"]
    # without the renumbering, or with the inverse permutation, the digest is another set's
    assert (oracle.cbo_digest(prows, n, m, threads=threads)["hsum"]) != want[0]
    inverse = np.argsort(perm)
    assert (oracle.cbo_digest(prows, n, m, threads=threads, label=inverse)["hsum"]) != want[0]
    with pytest.raises(RuntimeError):   # a label that is not a permutation is refused
        oracle.cbo_digest(prows, n, m, label=np.zeros(m, dtype=np.int32))


def test_extents_are_derivations():
    rows = cx.random_context(70, 40, 0.3, 9)
    r = oracle.cbo(rows, 70, 40, want_extents=True)
    ext_cells = cx.unpack_rows(r["extents"], 70)
    for i in range(r["intents"].shape[0]):
        assert np.array_equal(ext_cells[i], oracle.derive_extent(rows, r["intents"][i]))


# ---------------------------------------------------------------- mutation checks

MUTANTS = {
    "mask_includes_bit_j": ("return (d[full] & mask) == (b[full] & mask);",
                            "mask |= ((uint64_t)1) << (j & 63);\n    return (d[full] & mask) == (b[full] & mask);"),
    "no_saturation_skip": ("        if (bit_of(b, j)) continue;\n        s->closures += 1;",
                           "        s->closures += 1;"),
    "empty_extent_gives_nothing": ("    out[c->wm - 1] = c->last_attr_mask;          /* empty extent -> all M */",
                                   "    for (int32_t w = 0; w < c->wm; ++w) out[w] = 0;"),
    "child_cursor_skips_one": ("visit(c, s, stack, cc, dd, j + 1, depth + 1)",
                               "visit(c, s, stack, cc, dd, j + 2, depth + 1)"),
    "prefix_skips_word_0": ("for (int32_t w = 0; w < full; ++w)\n        if (d[w] != b[w]) return 0;",
                            "for (int32_t w = 1; w < full; ++w)\n        if (d[w] != b[w]) return 0;"),
    "or_instead_of_and": ("for (int64_t w = 0; w < c->wn; ++w) cc[w] = a[w] & col[w];",
                          "for (int64_t w = 0; w < c->wn; ++w) cc[w] = a[w] | col[w];"),
    "saturation_tests_extent": ("        if (bit_of(b, j)) continue;\n        s->closures += 1;",
                                "        if (bit_of(a, j)) continue;\n        s->closures += 1;"),
    "top_misses_last_object": ("for (int64_t o = 0; o < n; ++o) top_ext[o >> 6]",
                               "for (int64_t o = 0; o + 1 < n; ++o) top_ext[o >> 6]"),
    "mask_one_bit_short": ("(m % 64) ? ((((uint64_t)1) << (m % 64)) - 1u)",
                           "(m % 64) ? ((((uint64_t)1) << (m % 64 - 1)) - 1u)"),
}


def _quick_pins(lib):
    """Return the first pin that fails with this oracle build, or None."""
    for name in golden_names():
        n, m, rows, expected = load_golden(name)
        if not same_set(oracle.cbo(rows, n, m, lib=lib)["intents"], expected):
            return "golden " + name
    for n in (6, 9):
        if oracle.cbo(cx.contranominal(n), n, n, lib=lib)["intents"].shape[0] != 2 ** n:
            return "contranominal"
    r = oracle.cbo(cx.identity(70), 70, 70, lib=lib)
    if r["intents"].shape[0] != 72:
        return "identity"
    for (n, m, d, s) in [(33, 12, 0.3, 0), (20, 16, 0.5, 1)]:
        rows = cx.random_context(n, m, d, s)
        got = oracle.cbo(rows, n, m, lib=lib)["intents"]
        if has_duplicates(got) or not same_set(got, oracle.brute_force(rows, n, m)):
            return "brute force"
    for (n, m, d, s) in [(14, 100, 0.6, 6), (16, 70, 0.7, 3)]:
        rows = cx.random_context(n, m, d, s)
        got = oracle.cbo(rows, n, m, lib=lib)["intents"]
        if has_duplicates(got) or not same_set(got, oracle.brute_force_by_objects(rows, n, m)):
            return "object brute force"
    return None


def test_unmutated_oracle_passes_quick_pins():
    from oracle import cbo_binding as cbo_mod
    assert _quick_pins(cbo_mod.load()) is None


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant):
    from oracle import cbo_binding as cbo_mod
    src = open(os.path.join(os.path.dirname(oracle.__file__), "cbo.c")).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) >= 1, f"mutation site for {mutant} not found in the oracle source"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "cbo_mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new, 1))
        lib_path = cbo_mod.build_oracle(force=True, src=path, out=os.path.join(tmp, "libmut.so"))
        lib = cbo_mod.load(lib_path)
        assert _quick_pins(lib) is not None, f"mutant {mutant} passed every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


@pytest.mark.parametrize("n,m,p,seed", [(60, 10, 0.35, 3), (120, 14, 0.3, 4), (200, 9, 0.5, 5)])
def test_slice_identity_behind_the_full_size_checks(n, m, p, seed):
    """The intents containing S are the intents of the sub-context of the objects holding S (the
    identity the full-size slice checks rest on), on contexts small enough to enumerate whole."""
    rows = cx.random_context(n, m, p, seed)
    whole = oracle.cbo(rows, n, m)["intents"]
    for a in range(m):
        for b in (a, (a + 3) % m):
            mask = np.zeros(1, dtype=np.uint32)
            mask[0] = (1 << a) | (1 << b)
            inside = whole[(whole[:, 0] & mask[0]) == mask[0]]
            ext = oracle.derive_extent(rows, mask)
            sub = np.ascontiguousarray(rows[ext])
            if sub.shape[0] == 0:
                assert inside.shape[0] == 1      # only the bottom (every attribute) contains S
                continue
            ref = oracle.cbo(sub, sub.shape[0], m)["intents"]
            assert same_set(inside, ref)
