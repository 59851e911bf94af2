"""Host arithmetic of the benchmark's roofline (bench.py), checked by hand on made-up figures: the
bound is the slowest of HBM, HBM + L2 and word operations; achieved is the bound's quantity per
launch over the average launch time; the lean and the bitmap models use their own word counts."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_bound_picks_the_slowest(bench):
    # 1 GB of HBM at 1000 GB/s = 1 ms; 1 GB + 3 GB at 2000 GB/s = 2 ms; 1 Gop at 500 Gop/s = 2 ms
    r = bench.bound_of(1e9, 3e9, 1e9, 2, 4.0, 1000.0, "x", 2000.0, 250.0, 1, 1.0)
    assert r["bound"] == "alu"                      # 4 ms: the slowest
    assert r["bound_ms"] == pytest.approx({"hbm": 1.0, "l2": 2.0, "alu": 4.0})
    assert r["per_launch"] == pytest.approx(0.5e9)  # ops per launch (2 launches)
    assert r["achieved"] == pytest.approx(0.5e9 / 4e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 250.0)
    r = bench.bound_of(8e9, 0.0, 1e6, 1, 10.0, 1000.0, "x", 2000.0, 250.0, 1, 1.0)
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(8e9 / 10e-3 / 1e9 / 1000.0)


def test_roofline_uses_the_dominant_tier_and_both_models(bench, monkeypatch):
    tiers = {t: dict(parents=1, closures=2, children=3, isect_words=0, closure_words=0, canon_words=0,
                     hbm_words=0, hbm_lean_words=0, l2_lean_words=0) for t in ("list", "mid", "bitmap")}
    tiers["mid"].update(isect_words=100, closure_words=50, canon_words=10, hbm_words=1000,
                        hbm_lean_words=200, l2_lean_words=300)
    monkeypatch.setattr(bench, "load_work_counts", lambda *a: tiers)
    monkeypatch.setattr(bench, "profile_traffic", lambda *a: None)
    kms = {"subtree_kernel": 1.0, "expand_mid_kernel": 2.0, "expand_bitmap_kernel": 0.5}
    last = {"subtree_launches": 1, "mid_launches": 4, "expand_launches": 1, "mid_max": 256, "list_max": 1000}
    counted = {"subtree_word_ops": 0, "expand_bytes": 0, "subtree_launches": 1, "expand_launches": 1}
    r = bench.roofline_of("w", "support", kms, last, counted, {"l2_read_gbs": 1e-6}, {"hbm_gbs": 1e-6}, 1, 1.0)
    assert r["kernel"] == "expand_mid_kernel" and r["launches_per_step"] == 4
    assert r["avg_launch_ms"] == pytest.approx(0.5)
    # lean: HBM 800 B, L2 1200 B: (800 + 1200) B at 1e-6 GB/s is the slowest bound
    assert r["bound"] == "l2" and r["per_launch"] == pytest.approx(2000.0 / 4)
    # bitmap model: HBM 4000 B, L2 600 B
    assert r["bitmap_model"]["per_launch"] == pytest.approx(4600.0 / 4)
    assert r["units_per_step"] == {"parents": 1, "closures": 2, "children": 3}


def test_cover_counts_are_stored_and_consistent(bench):
    """The cover-search work counts that the covers stage divides by its time are stored for the
    workloads it is run on, with one concept per intent of the stored digests and the intersection
    words at most (M - 0) x W_N per concept (every attribute outside B over at most every word)."""
    import json
    digests = json.load(open(os.path.join(ROOT, "tests", "golden", "workload_digests.json")))
    for name in ("sparse", "zipf", "skewed"):
        cw = bench.load_cover_counts(name)
        assert cw is not None, name
        d = digests[name]
        assert cw["concepts"] == d["concepts"]
        wn = (d["n_objects"] + 31) // 32
        assert cw["extent_words"] == cw["concepts"] * wn
        assert 0 < cw["isect_words"] <= cw["concepts"] * d["n_attrs"] * wn
        assert cw["closure_words"] > 0
    assert bench.load_cover_counts("no such workload") is None
