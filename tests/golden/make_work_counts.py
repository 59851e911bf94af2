"""Write tests/golden/work_counts.json from the work-counting pass in oracle/ (and nothing else).

For each named synthetic workload it records, per tier of parent extent (at most 64 objects:
"list"; more: "bitmap"), the algorithmic work of the whole enumeration in 32-bit words: parents,
closures, canonical children, extent-intersection words, closure words (the cheaper of the row and
column routes), canonical-test words and HBM words (extent reads, frontier and output writes).
The benchmark divides these by measured kernel time for its roofline figures. The search runs over
the table in the library's default processing order (ascending attribute support), the order in
which the kernels do their work; --order natural counts the attribute order instead.

usage: python tests/golden/make_work_counts.py [workload ...] [--threads T] [--order support|natural]
"""
import argparse
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from oracle.workcount import workcount  # noqa: E402
from closed_set_enumeration_gb300 import contexts as cx  # noqa: E402
from tests._util import support_order  # noqa: E402

OUT = os.path.join(HERE, "work_counts.json")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("names", nargs="*", default=["tiny", "sparse", "zipf", "skewed"])
    ap.add_argument("--threads", type=int, default=os.cpu_count() or 1)
    ap.add_argument("--order", choices=["support", "natural"], default="support")
    args = ap.parse_args()
    for name in args.names:
        w = cx.WORKLOADS[name]
        rows = w.rows()
        if args.order == "support":
            rows = support_order(rows, w.n_objects, w.n_attrs)[0]
        t0 = time.time()
        counts = workcount(rows, w.n_objects, w.n_attrs, threads=args.threads)
        dt = time.time() - t0
        # re-read before writing: several runs may fill in different workloads
        data = json.load(open(OUT)) if os.path.exists(OUT) else {}
        data[name] = {"n_objects": w.n_objects, "n_attrs": w.n_attrs, "seed": w.seed, "tiers": counts,
                      "order": args.order, "seconds": round(dt, 1), "threads": args.threads}
        with open(OUT + ".tmp", "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)
            f.write("\n")
        os.replace(OUT + ".tmp", OUT)
        print(name, f"{dt:.1f}s", counts, flush=True)


if __name__ == "__main__":
    main()
