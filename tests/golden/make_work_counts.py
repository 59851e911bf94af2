"""Write tests/golden/work_counts.json from the work-counting pass in oracle/ (and nothing else).

For each named synthetic workload it records, per tier of parent extent (at most 64 objects:
"list"; at most --mid-max objects: "mid"; more: "bitmap"), the algorithmic work of the whole enumeration in 32-bit words: parents,
closures, canonical children, extent-intersection words, closure words (the cheaper of the row and
column routes), canonical-test words and HBM words (extent reads, frontier and output writes).
The benchmark divides these by measured kernel time for its roofline figures. The search runs over
the table in the library's default processing order (ascending attribute support), the order in
which the kernels do their work; --order natural counts the attribute order instead.

The mid-tier bound is the largest extent the library expands one search node per warp, and the
list bound the largest extent it keeps as an object-id list (its statistics report them as mid_max
and list_max: 256, and 315 / 928 / 1312 objects for the skewed / zipf / planted-bicluster tables;
none for the two smaller ones); they are given on the command line, so that this script calls only
oracle/. The list bound enters only the lean model's fields (hbm_lean_words, l2_lean_words).

With --covers it records instead, under the workload's "covers" key, the work of the lower-cover
search over the workload's whole intent set (oracle/coverwork.c: per concept its extent, the
intersections A & column k for k outside B, and the closure of each non-empty one by rows), over
the intents the oracle enumerates; the count does not depend on their order.

usage: python tests/golden/make_work_counts.py [workload ...] [--threads T] [--order support|natural]
                                               [--mid-max T] [--list-max L] [--covers]
"""
import argparse
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle.workcount import coverwork, workcount  # noqa: E402
from closed_set_enumeration_gb300 import contexts as cx  # noqa: E402
from tests._util import support_order  # noqa: E402

OUT = os.path.join(HERE, "work_counts.json")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("names", nargs="*", default=["tiny", "sparse", "zipf", "skewed"])
    ap.add_argument("--threads", type=int, default=os.cpu_count() or 1)
    ap.add_argument("--order", choices=["support", "natural"], default="support")
    ap.add_argument("--mid-max", type=int, default=0, help="largest extent of the mid tier (0: none)")
    ap.add_argument("--list-max", type=int, default=0, help="largest extent kept as an id list (0: none)")
    ap.add_argument("--covers", action="store_true", help="count the lower-cover search instead")
    args = ap.parse_args()
    if args.covers:
        for name in args.names:
            w = cx.WORKLOADS[name]
            rows = w.rows()
            t0 = time.time()
            intents = oracle.cbo(rows, w.n_objects, w.n_attrs, threads=args.threads)["intents"]
            counts = coverwork(rows, w.n_objects, w.n_attrs, intents, threads=args.threads)
            dt = time.time() - t0
            data = json.load(open(OUT)) if os.path.exists(OUT) else {}
            data.setdefault(name, {})["covers"] = dict(counts, seconds=round(dt, 1), threads=args.threads)
            with open(OUT + ".tmp", "w") as f:
                json.dump(data, f, indent=1, sort_keys=True)
                f.write("\n")
            os.replace(OUT + ".tmp", OUT)
            print(name, "covers", f"{dt:.1f}s", counts, flush=True)
        return
    for name in args.names:
        w = cx.WORKLOADS[name]
        rows = w.rows()
        if args.order == "support":
            rows = support_order(rows, w.n_objects, w.n_attrs)[0]
        t0 = time.time()
        counts = workcount(rows, w.n_objects, w.n_attrs, threads=args.threads, mid_max=args.mid_max,
                           list_max=args.list_max)
        dt = time.time() - t0
        # re-read before writing: several runs may fill in different workloads
        data = json.load(open(OUT)) if os.path.exists(OUT) else {}
        covers = data.get(name, {}).get("covers")
        data[name] = {"n_objects": w.n_objects, "n_attrs": w.n_attrs, "seed": w.seed, "tiers": counts,
                      "order": args.order, "mid_max": args.mid_max, "list_max": args.list_max,
                      "seconds": round(dt, 1),
                      "threads": args.threads}
        if covers is not None:
            data[name]["covers"] = covers
        with open(OUT + ".tmp", "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)
            f.write("\n")
        os.replace(OUT + ".tmp", OUT)
        print(name, f"{dt:.1f}s", counts, flush=True)


if __name__ == "__main__":
    main()
