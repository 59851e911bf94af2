"""Full-size workloads, checked where the oracle cannot enumerate the whole context in test time.

The intents of a context K that contain an attribute set S are exactly the intents of the
sub-context K[S'] made of the objects that hold all of S (every attribute set closed in K[S'] is
the AND of some of its rows, or M, and the derivation of an extent inside S' is the same in K and
in K[S']). So the slice of the GPU's full-size output made of the intents containing S must equal,
as a set, the oracle's enumeration of K[S'] — an exact check of a part of the full launch that the
oracle finishes in seconds. Besides the slices, every full-size output is checked for properties
that hold at any size: no duplicates, the top and bottom intents present, fixed points B'' = B of
sampled intents (the oracle's derivation operators, one intent at a time), and closure of the set
under intersection on sampled pairs.
"""
import numpy as np
import pytest

import oracle
from closed_set_enumeration_gb300 import build as fbuild
from closed_set_enumeration_gb300 import contexts as cx
from tests._util import sort_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fbuild.build()


def _row_keys(t, torch):
    """A 63-bit mix of each intent row (device), for sorting and membership tests."""
    h = torch.zeros(t.shape[0], dtype=torch.int64, device=t.device)
    for w in range(t.shape[1]):
        v = t[:, w].to(torch.int64) & 0xFFFFFFFF
        h = (h * 0x100000001B3 + v * 0x9E3779B1 + w) & 0x7FFFFFFFFFFFFFFF
    return h


def _choose_slices(rows, n_attrs, lo, hi, count):
    """Attribute sets S (single attributes, then pairs) whose extents S' hold between lo and hi
    objects, chosen in attribute order."""
    chosen = []
    cols = [(rows[:, a >> 5] >> np.uint32(a & 31)) & np.uint32(1) for a in range(n_attrs)]
    for a in range(n_attrs):
        s = int(cols[a].sum())
        if lo <= s <= hi:
            chosen.append((a,))
        if len(chosen) == count:
            return chosen
    for a in range(n_attrs):
        for b in range(a + 1, n_attrs):
            s = int((cols[a] & cols[b]).sum())
            if lo <= s <= hi:
                chosen.append((a, b))
            if len(chosen) == 2 * count:
                return chosen
    return chosen


SLICE_CASES = {
    # workload: (min |S'|, max |S'|, slices)
    "sparse": (150, 400, 3),
    "skewed": (200, 1500, 3),
    "zipf": (300, 3000, 3),
    "biclusters": (500, 3000, 3),
}


@pytest.mark.parametrize("name", list(SLICE_CASES))
def test_full_size_slices_and_properties(name):
    import torch
    from closed_set_enumeration_gb300 import fca

    w = cx.WORKLOADS[name]
    rows = w.rows()
    wm = (w.n_attrs + 31) // 32
    with fca.Context(rows, w.n_objects, w.n_attrs) as ctx:
        out = ctx.enumerate()                       # device tensor (K, W_M), int32 words
    K = out.shape[0]
    assert K > 0

    # no duplicates: sort by one mix, compare the rows of equal mixes word by word
    h1 = _row_keys(out, torch)
    order = torch.argsort(h1)
    s1 = h1[order]
    del h1
    same = torch.nonzero(s1[1:] == s1[:-1]).flatten()
    if same.numel():
        a, b = order[same], order[same + 1]
        assert not bool((out[a] == out[b]).all(dim=1).any()), "duplicate intents"

    # the top intent (AND of all rows) and the bottom (every attribute) are present
    def present(row):
        r = torch.from_numpy(np.asarray(row, dtype=np.uint32).view(np.int32)).to(out.device)
        k1 = _row_keys(r[None, :], torch)
        pos = torch.searchsorted(s1, k1)
        lo = int(pos[0])
        while lo < K and int(s1[lo]) == int(k1[0]):
            if bool((out[order[lo]] == r).all()):
                return True
            lo += 1
        return False

    top = np.bitwise_and.reduce(rows, axis=0)
    full = np.full(wm, 0xFFFFFFFF, dtype=np.uint32)
    if w.n_attrs & 31:
        full[-1] = (1 << (w.n_attrs & 31)) - 1
    top &= full
    assert present(top)
    assert present(full)

    # fixed points of sampled intents, one by one
    rng = np.random.default_rng(1)
    idx = rng.choice(K, size=min(K, 100), replace=False)
    host = out[torch.from_numpy(idx).to(out.device)].cpu().numpy().view(np.uint32)
    for b in host:
        ext = oracle.derive_extent(rows, b)
        assert np.array_equal(oracle.derive_intent(rows, ext, w.n_attrs), b)

    # closure under intersection, on sampled pairs
    pairs = rng.choice(K, size=(100, 2))
    pa = out[torch.from_numpy(pairs[:, 0]).to(out.device)]
    pb = out[torch.from_numpy(pairs[:, 1]).to(out.device)]
    for r in (pa & pb).cpu().numpy().view(np.uint32):
        assert present(r), "intersection of two intents is not an intent"

    # slices: intents containing S equal the oracle's intents of the sub-context K[S']
    lo_s, hi_s, count = SLICE_CASES[name]
    slices = _choose_slices(rows, w.n_attrs, lo_s, hi_s, count)
    assert slices, "no attribute set with a suitable extent size"
    for S in slices:
        mask = np.zeros(wm, dtype=np.uint32)
        for a in S:
            mask[a >> 5] |= np.uint32(1) << np.uint32(a & 31)
        m_dev = torch.from_numpy(mask.view(np.int32)).to(out.device)
        sel = out[((out & m_dev) == m_dev).all(dim=1)].cpu().numpy().view(np.uint32)
        ext = oracle.derive_extent(rows, mask)
        sub = np.ascontiguousarray(rows[ext])
        ref = oracle.cbo(sub, sub.shape[0], w.n_attrs, threads=4)["intents"]
        assert sel.shape[0] == ref.shape[0], f"slice {S}: {sel.shape[0]} intents, oracle {ref.shape[0]}"
        assert np.array_equal(sort_rows(sel), sort_rows(ref)), f"slice {S} differs from the oracle"
