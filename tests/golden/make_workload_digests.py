"""Write tests/golden/workload_digests.json from the CPU oracle (and nothing else).

For each named synthetic workload it records the number of intents, the
number of closures (candidates evaluated by Close-by-One), the concepts per
search depth, an order-independent digest of the intent set (sum and xor mod
2^64 of one hash per intent, computed by the oracle's digest mode) and, when
the intents fit in host memory, a SHA-256 digest of the intents sorted as big
integers (last 32-bit word most significant), so that full-size GPU runs can
be checked without re-running the oracle. It also records the closures of the
same search over the table in ascending-support attribute order (the library's
default processing order; the intent set is the same), with --order-closures
alone without redoing the rest. That search also digests its intents renumbered
back to the original attributes, which gives the multiset digest of a workload
whose search in attribute order is too long for the host.

usage: python tests/golden/make_workload_digests.py [workload ...] [--threads T] [--digest-only]
                                                    [--order-closures]
"""
import argparse
import hashlib
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from closed_set_enumeration_gb300 import contexts as cx  # noqa: E402
from tests._util import support_order  # noqa: E402

OUT = os.path.join(HERE, "workload_digests.json")


def digest(intents: np.ndarray) -> str:
    rows = np.ascontiguousarray(intents, dtype="<u4")
    rows = rows[np.lexsort(rows.T)] if rows.shape[0] else rows
    return hashlib.sha256(np.ascontiguousarray(rows).tobytes()).hexdigest()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("names", nargs="*", default=list(cx.WORKLOADS))
    ap.add_argument("--threads", type=int, default=os.cpu_count() or 1)
    ap.add_argument("--digest-only", action="store_true", help="skip the sorted SHA-256 (large sets)")
    ap.add_argument("--order-closures", action="store_true",
                    help="only (re)compute the closures in ascending-support order")
    args = ap.parse_args()
    data = json.load(open(OUT)) if os.path.exists(OUT) else {}
    for name in args.names:
        w = cx.WORKLOADS[name]
        rows = w.rows()
        t0 = time.time()
        prows, inv = support_order(rows, w.n_objects, w.n_attrs)
        go = oracle.cbo_digest(prows, w.n_objects, w.n_attrs, threads=args.threads, label=inv)
        if args.order_closures:
            data = json.load(open(OUT)) if os.path.exists(OUT) else {}
            entry = data.get(name, {})
            if "concepts" in entry:
                assert entry["concepts"] == go["count"]
            else:   # a workload whose search in attribute order is too long for the host
                entry.update({"n_objects": w.n_objects, "n_attrs": w.n_attrs, "seed": w.seed,
                              "concepts": go["count"], "oracle_order": "support",
                              "oracle_seconds": round(time.time() - t0, 1), "oracle_threads": args.threads})
            entry["closures_support_order"] = go["closures"]
            hs, hx = f"{go['hsum']:016x}", f"{go['hxor']:016x}"
            if "multiset_hsum" in entry:
                assert (entry["multiset_hsum"], entry["multiset_hxor"]) == (hs, hx)
            else:
                entry.update({"multiset_hsum": hs, "multiset_hxor": hx, "digest_search_order": "support"})
            data[name] = entry
            print(name, "support order", go["count"], go["closures"], f"{time.time() - t0:.1f}s", flush=True)
            with open(OUT, "w") as f:
                json.dump(data, f, indent=1, sort_keys=True)
            continue
        t0 = time.time()
        g = oracle.cbo_digest(rows, w.n_objects, w.n_attrs, threads=args.threads)
        dt = time.time() - t0
        depth = [int(x) for x in g["depth_counts"]]
        while depth and depth[-1] == 0:
            depth.pop()
        entry = (json.load(open(OUT)) if os.path.exists(OUT) else {}).get(name, {})
        entry.update({
            "n_objects": w.n_objects, "n_attrs": w.n_attrs, "seed": w.seed,
            "concepts": g["count"], "closures": g["closures"], "depth_counts": depth,
            "multiset_hsum": f"{g['hsum']:016x}", "multiset_hxor": f"{g['hxor']:016x}",
            "oracle_seconds": round(dt, 1), "oracle_threads": args.threads,
            "closures_support_order": go["closures"],
        })
        # the intent set does not depend on the order of the search
        assert (g["hsum"], g["hxor"]) == (go["hsum"], go["hxor"])
        if not args.digest_only:
            r = oracle.cbo(rows, w.n_objects, w.n_attrs, threads=args.threads)
            assert r["intents"].shape[0] == g["count"] and r["closures"] == g["closures"]
            entry["sha256_sorted_intents"] = digest(r["intents"])
        # re-read before writing: several runs (one per workload) may update the file
        data = json.load(open(OUT)) if os.path.exists(OUT) else {}
        data[name] = entry
        print(name, data[name]["concepts"], data[name]["closures"], f"{dt:.1f}s", flush=True)
        with open(OUT, "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
