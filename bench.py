#!/usr/bin/env python
"""Throughput of full formal-concept enumeration on GB300.

One step = one pass of the whole hot path over one synthetic context: load the
rows into the context (row copy, padding mask, transpose to columns, top
intent) and enumerate every intent (bitmap- and mid-tier expansion, object-list
subtrees, compaction into the output buffer). Inputs are resident in device
memory when the timed region starts; L2 is flushed between timed steps. The
default workload is the largest one that fits one GPU, the planted-bicluster
table (100 000 x 256, 519 340 217 concepts).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0). With N > 1 (torchrun), every rank enumerates its
own copy of the workload (independent replicas, no collective on the data
path); value = concepts of all ranks / slowest rank's time. The timed steps
reuse the context's work pools; `first_call_ms` is the first enumeration on a
fresh context (pools allocated and levels planned inside the call), reported
beside them.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from closed_set_enumeration_gb300 import contexts as cx  # noqa: E402

METRIC = "concepts/sec (closures/sec) per GB300; fraction of bitwise INT/L2 roofline"
UNIT = "concepts/s"
DEFAULT_WORKLOAD = "biclusters"
L2_FLUSH_BYTES = 512 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
INT_LANES_PER_SM = 64        # 32-bit logical-op results per SM per clock (checked by the LOP3 probe)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(cx.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="budget of the CPU oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--lattice-rows", type=int, default=0,
                    help="extents / covers stages: only the first R intents (0: all; covers needs all)")
    ap.add_argument("--stage", choices=["enumerate", "extents", "covers"], default="enumerate",
                    help="enumerate: the intents (the default line); extents / covers: the lattice calls "
                         "on the workload's intents, timed alone")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle baseline

class OracleSampler:
    """Concepts/s of the CPU oracle (test infrastructure) on a bounded sample of a workload.

    A sample is either whole enumerations of the workload, repeated until the time budget is
    used, or - when one enumeration would not fit the budget - one enumeration whose threads stop
    after a fixed number of intents each (the limit is calibrated once to fit the budget).
    """

    def __init__(self, rows, w, threads: int):
        import oracle
        self.oracle = oracle
        self.rows, self.w, self.threads = rows, w, threads
        self.limit = None
        oracle.cbo(cx.random_context(40, 12, 0.3, 0), 40, 12)   # build/load outside any timing

    def _run(self, limit: int):
        t0 = time.perf_counter()
        r = self.oracle.cbo(self.rows, self.w.n_objects, self.w.n_attrs, threads=self.threads, limit=limit)
        return int(r["intents"].shape[0]), time.perf_counter() - t0

    def sample(self, budget_s: float):
        if self.limit is None:
            cnt, dt = self._run(0) if self._fits(budget_s) else (None, None)
            if cnt is not None:
                self.limit = 0
            else:
                lim = 4096
                while True:
                    cnt, dt = self._run(lim)
                    if dt >= budget_s / 4 or lim >= 1 << 28:
                        break
                    lim *= 4
                self.limit = lim
                return cnt / dt, f"one enumeration stopped after {lim} intents per thread", dt
        if self.limit:
            cnt, dt = self._run(self.limit)
            return cnt / dt, f"one enumeration stopped after {self.limit} intents per thread", dt
        total, runs, t0 = 0, 0, time.perf_counter()
        while True:
            cnt, _ = self._run(0)
            total += cnt
            runs += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                return total / el, f"{runs} whole enumeration(s) of the workload", el

    def _fits(self, budget_s: float) -> bool:
        digests = os.path.join(ROOT, "tests", "golden", "workload_digests.json")
        try:
            d = json.load(open(digests)).get(self.w.name) or {}
        except (OSError, ValueError):
            d = {}
        full_s = d.get("oracle_seconds")
        return full_s is not None and full_s * d.get("oracle_threads", 1) / max(1, self.threads) < budget_s


def cpu_baseline(rows, w, budget_s: float):
    """The oracle on all host cores (the top-level attributes split between threads) and, beside
    it, on one thread (the single-thread form of the pages' CPU baseline), each on a bounded
    sample of the workload."""
    threads = os.cpu_count() or 1
    rate, sample, dt = OracleSampler(rows, w, threads).sample(budget_s)
    rate1, sample1, dt1 = OracleSampler(rows, w, 1).sample(max(1.0, budget_s / 2))
    return {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
            "seconds": round(dt, 2),
            "single_thread": {"value": rate1, "unit": UNIT, "cores": 1, "sample": sample1,
                              "seconds": round(dt1, 2)}}


# ----------------------------------------------------------------------------- roofline helpers

# The source file of each kernel a roofline is reported for.
KERNEL_SOURCES = {"subtree_kernel": "fca_subtree.cuh", "expand_bitmap_kernel": "fca_expand.cu",
                  "expand_mid_kernel": "fca_mid.cu", "extents_kernel": "fca_lattice.cu",
                  "covers_kernel": "fca_lattice.cu"}


def profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summary, or None.

    The summary records the SHA-256 of the kernel source it was taken on; once the source has
    changed the figure no longer applies and None is returned.
    """
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, "closed_set_enumeration_gb300", "csrc", KERNEL_SOURCES[kernel])
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-* ").replace("`", "")
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256") != sha:
        return None
    try:
        return float(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def profile_traffic_per_row(kernel: str, workload: str):
    """DRAM bytes per processed row of `kernel` on `workload` from its committed ncu summary (the
    capture's traffic over its rows), or None once the kernel source has changed."""
    t = profile_traffic(kernel, workload)
    if t is None:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")).read()
        rows = [ln.split(":", 1)[1] for ln in text.splitlines() if ln.strip().lstrip("-* ").startswith("rows_per_launch:")]
        return t / float(rows[0].strip().replace(",", ""))
    except (OSError, IndexError, ValueError):
        return None


def load_peaks():
    try:
        return json.load(open(PEAKS_FILE))
    except (OSError, ValueError):
        return None


def probe_peaks():
    """LOP3 issue rate and L2 read bandwidth measured on this GPU by the probe library."""
    import ctypes
    path = os.path.join(ROOT, "closed_set_enumeration_gb300", "libfca_probe.so")
    lib = ctypes.CDLL(path)
    lib.fca_probe_lop3.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.fca_probe_read_bw.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    ops, ms, l2 = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    out = {}
    if lib.fca_probe_lop3(ctypes.byref(ops), ctypes.byref(ms)) == 0:
        out["lop3_gops"] = ops.value / 1e9
    if lib.fca_probe_read_bw(16 << 20, 5, ctypes.byref(l2)) == 0:
        out["l2_read_gbs"] = l2.value
    return out


WORK_FILE = os.path.join(ROOT, "tests", "golden", "work_counts.json")


def load_cover_counts(workload: str):
    """Work of the lower-cover search over a workload's intent set, written by
    tests/golden/make_work_counts.py --covers, or None."""
    try:
        return json.load(open(WORK_FILE))[workload].get("covers")
    except (OSError, ValueError, KeyError):
        return None


def load_work_counts(workload: str, order: str, mid_max: int, list_max: int):
    """Per-tier algorithmic work of a workload, written by tests/golden/make_work_counts.py, when it
    was counted over the attribute order the library processes ("natural" or "support") and with
    the library's tier split and id-list bound."""
    try:
        entry = json.load(open(WORK_FILE))[workload]
    except (OSError, ValueError, KeyError):
        return None
    if (entry.get("order", "natural") != order or int(entry.get("mid_max", 0)) != int(mid_max)
            or int(entry.get("list_max", 0)) != int(list_max)):
        return None
    return entry.get("tiers")


# the kernel of each tier: parents of at most 64 objects, of at most mid_max, and larger
TIER_KERNELS = (("list", "subtree_kernel", "subtree_ms", "subtree_launches"),
                ("mid", "expand_mid_kernel", "mid_ms", "mid_launches"),
                ("bitmap", "expand_bitmap_kernel", "expand_ms", "expand_launches"))


def bound_of(hbm_b, l2_b, ops, nl, avg_ms, hbm_peak, hbm_basis, l2_peak, int_peak, sm_count, sm_max):
    """The slowest of HBM bytes at the measured copy bandwidth, HBM + L2 bytes at the probed L2 read
    bandwidth and word operations at the int32 issue rate; achieved = the bound's quantity per
    launch over the average launch time."""
    times = {"hbm": hbm_b / (hbm_peak * 1e9), "l2": (hbm_b + l2_b) / (l2_peak * 1e9), "alu": ops / (int_peak * 1e9)}
    bound = max(times, key=times.get)
    if bound == "alu":
        per_launch, unit, peak, basis = ops / nl, "Gop/s", int_peak, \
            f"{sm_count} SMs x {INT_LANES_PER_SM} int32 lanes x {sm_max:.0f} MHz"
    elif bound == "hbm":
        per_launch, unit, peak, basis = hbm_b / nl, "GB/s", hbm_peak, hbm_basis
    else:
        per_launch, unit, peak, basis = (hbm_b + l2_b) / nl, "GB/s", l2_peak, \
            "L2 read probe in this run (16 MiB buffer re-read)"
    achieved = per_launch / (avg_ms * 1e-3) / 1e9
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "peak_basis": basis, "per_launch": per_launch, "bound_ms": {k: v * 1e3 for k, v in times.items()}}


def roofline_of(workload, order, kernel_ms, last, counted, probes, peaks, sm_count, sm_max):
    """Roofline of the kernel with the largest device time per step.

    The numerator is the algorithmic work of that kernel's tier (parents of at most 64 objects run
    in subtree_kernel, those of at most mid_max objects in expand_mid_kernel, larger ones in
    expand_bitmap_kernel), counted exactly by the CPU counting pass. Two models of the words moved:
    the method's (every search node's extent an N-bit bitmap read once, every child's written) and
    the lean one of this library's representation (extents of at most list_max objects as id lists,
    object-list subtrees searched in place, rows gathered once per parent kept as a list). The
    roofline reported is the lean model's, the tighter bound for these kernels; the bitmap model's
    figures come beside it. Either bound is the slowest of HBM bytes at the measured copy bandwidth,
    HBM + L2 bytes at the L2 read bandwidth probed in this run, and word operations at the int32
    issue rate (SMs x 64 lanes x maximum SM clock); achieved / peak is the bound's time over the
    measured kernel time (the union of the launches' intervals, per step). Without stored counts
    for the workload in the library's processing order and tier split, the kernel's own counted
    work (the counting launch) stands in for the object-list tier, and `basis` says so.
    """
    tier, kernel, _, launches_key = max(TIER_KERNELS, key=lambda t: kernel_ms[t[1]])
    kms = kernel_ms[kernel]
    nl = max(1, last[launches_key])
    avg_ms = kms / nl
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    hbm_basis = "MEASURED_PEAKS.json hbm_gbs" if "hbm_gbs" in peaks else "fallback 6.8 TB/s"
    l2_peak = probes.get("l2_read_gbs") or hbm_peak
    int_peak = sm_count * INT_LANES_PER_SM * sm_max * 1e6 / 1e9   # Gop/s
    out = {"kernel": kernel, "avg_launch_ms": avg_ms, "launches_per_step": nl,
           "traffic": profile_traffic(kernel, workload)}
    work = load_work_counts(workload, order, last.get("mid_max", 0), last.get("list_max", 0))
    args = (nl, avg_ms, hbm_peak, hbm_basis, l2_peak, int_peak, sm_count, sm_max)
    if work is not None and tier in work and "hbm_lean_words" in work[tier]:
        t = work[tier]
        ops = t["isect_words"] + t["closure_words"] + t["canon_words"]
        out.update(bound_of(4.0 * t["hbm_lean_words"], 4.0 * t["l2_lean_words"], ops, *args))
        out["basis"] = "algorithmic work of the tier, lean model (oracle/workcount.c)"
        out["bitmap_model"] = bound_of(4.0 * t["hbm_words"], 4.0 * (t["isect_words"] + t["closure_words"]), ops, *args)
        out["units_per_step"] = {"parents": t["parents"], "closures": t["closures"], "children": t["children"]}
    elif tier == "list":
        per_launch = counted["subtree_word_ops"] / max(1, counted["subtree_launches"])
        achieved = per_launch / (avg_ms * 1e-3) / 1e9
        out.update({"bound": "alu", "achieved": achieved, "peak": int_peak, "unit": "Gop/s",
                    "frac": achieved / int_peak, "per_launch": per_launch,
                    "peak_basis": f"{sm_count} SMs x {INT_LANES_PER_SM} int32 lanes x {sm_max:.0f} MHz",
                    "basis": "word operations counted by the kernel (counting launch)"})
    else:
        out.update({"bound": None, "achieved": None, "peak": None, "frac": None,
                    "basis": "no stored work counts for this workload, order and tier split"})
    # the kernel's own counted work, for reference
    out["kernel_counted"] = {"subtree_word_ops": counted["subtree_word_ops"],
                             "expand_bytes": counted["expand_bytes"]}
    out["probe_lop3_gops"] = probes.get("lop3_gops")
    return out


# ----------------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import torch
    from closed_set_enumeration_gb300 import build as fbuild
    from closed_set_enumeration_gb300 import fca

    fbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = cx.WORKLOADS[args.workload]
    rows = w.rows()
    wm = (w.n_attrs + 31) // 32
    rows_dev = torch.from_numpy(rows.view(np.int32)).to(dev)
    stream = torch.cuda.current_stream(dev)

    ctx = fca.Context(rows_dev, w.n_objects, w.n_attrs)
    # the processing order the library chose for this table (see FCA_OPT_ATTR_ORDER)
    attr_order = "natural" if np.array_equal(ctx.copy_layout("order"), np.arange(w.n_attrs)) else "support"
    # one untimed counting pass: the algorithmic work of each kernel, and the exact output size
    ctx.set_option(fca.FCA_OPT_COUNT_WORK, 1)
    first = ctx.enumerate(stream=stream)
    counted = ctx.stats()
    ctx.set_option(fca.FCA_OPT_COUNT_WORK, 0)
    concepts = int(first.shape[0])
    del first
    out = torch.empty((concepts, wm), dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    table_kernels = 2 + (1 if w.n_attrs % 32 else 0)

    def step():
        ctx.load(rows_dev, stream=stream)
        st, cnt = ctx.enumerate_into(out, concepts, stream=stream)
        if st != fca.FCA_OK or cnt != concepts:
            raise RuntimeError(f"enumeration returned status {st}, count {cnt} (expected {concepts})")

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    step_ms, launches = [], 0
    kernel_ms = {k: 0.0 for _, k, _, _ in TIER_KERNELS}
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    for _ in range(args.steps):
        flush.zero_()                         # L2 flush between timed steps (outside the events)
        ev0.record(stream)
        step()
        ev1.record(stream)
        ev1.synchronize()
        step_ms.append(ev0.elapsed_time(ev1))
        s = ctx.stats()
        for _, k, ms_key, _ in TIER_KERNELS:
            kernel_ms[k] += s[ms_key]
        launches += s["launches"] + table_kernels
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    last = ctx.stats()

    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    value = concepts * args.steps * world / total_s
    closures_per_s = last["closures"] * args.steps * world / total_s

    # ---- end to end through the C ABI with host buffers: H2D of the rows, D2H of the intents
    pin_rows = torch.from_numpy(rows.view(np.int32)).pin_memory()
    pin_out = torch.empty((concepts, wm), dtype=torch.int32).pin_memory()
    pin_out_np = pin_out.numpy().view(np.uint32)
    e2e_steps = max(1, args.e2e_steps)
    for _ in range(2):
        ctx.load(pin_rows, stream=stream)
        ctx.enumerate_host(pin_out_np, stream=stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ctx.load(pin_rows, stream=stream)
        st, cnt = ctx.enumerate_host(pin_out_np, stream=stream)
        if cnt != concepts:
            raise RuntimeError("end-to-end count mismatch")
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    barrier(world)

    # ---- roofline of the dominant kernel
    probes = probe_peaks() if rank == 0 else {}
    peaks = load_peaks() or {}
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    steps = args.steps
    per_step = {k: v / steps for k, v in kernel_ms.items()}
    roofline = roofline_of(w.name, attr_order, per_step, last, counted, probes, peaks, sm_count, sm_max)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": total_s * 1e3 / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": w.name, "n_objects": w.n_objects, "n_attrs": w.n_attrs, "seed": w.seed,
                   "description": w.description, "concepts": concepts, "closures": last["closures"],
                   "attr_order": attr_order,
                   "l2": "flushed between timed steps (512 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "closures_per_s": closures_per_s,
        "e2e": {"value": concepts * e2e_steps * world / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": int(rows.nbytes), "d2h_bytes_per_step": int(concepts * wm * 4)},
        "gpu_launches": launches,
        "kernel_ms_per_step": per_step,
        "tiers": {"list_max": last["list_max"], "mid_max": last["mid_max"],
                  "large_parents": last["large_parents"], "small_roots": last["small_roots"]},
        "roofline": roofline,
        "clocks": clocks,
        "probes": probes,
    }
    # the first call on a fresh context (the work pools allocated and the levels planned inside the
    # call), which a caller with a new table pays once; the timed steps reuse the context's pools
    ctx.close()
    del pin_out, pin_out_np
    torch.cuda.synchronize(dev)
    fresh = fca.Context(rows_dev, w.n_objects, w.n_attrs)
    torch.cuda.synchronize(dev)
    t_first = time.perf_counter()
    fresh.enumerate_into(out, concepts, stream=stream)
    torch.cuda.synchronize(dev)
    result["first_call_ms"] = (time.perf_counter() - t_first) * 1e3
    fresh.close()
    return result


def run_lattice(args, world, rank, local):
    """Time fca_extents or fca_cover_edges on the workload's complete intent set (enumerated once,
    untimed), one call per step, with the L2 flushed between steps."""
    import torch
    from closed_set_enumeration_gb300 import build as fbuild
    from closed_set_enumeration_gb300 import fca

    fbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = cx.WORKLOADS[args.workload]
    rows = w.rows()
    wm, wn = (w.n_attrs + 31) // 32, (w.n_objects + 31) // 32
    stream = torch.cuda.current_stream(dev)
    ctx = fca.Context(torch.from_numpy(rows.view(np.int32)).to(dev), w.n_objects, w.n_attrs)
    intents = ctx.enumerate(stream=stream)
    if args.lattice_rows > 0 and args.stage == "extents":
        intents = intents[: args.lattice_rows]
    k = int(intents.shape[0])
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    if args.stage == "extents":
        out = torch.empty((k, wn), dtype=torch.int32, device=dev)

        def step():
            ctx.extents_into(intents, out, stream=stream)
        launches_per_step = 1
    else:
        edges = ctx.cover_edges(intents, stream=stream)
        n_edges = int(edges.shape[0])
        buf = torch.empty((n_edges, 2), dtype=torch.int32, device=dev)

        def step():
            st, cnt = ctx.cover_edges_into(intents, buf, n_edges, stream=stream)
            if st != fca.FCA_OK or cnt != n_edges:
                raise RuntimeError(f"fca_cover_edges returned {st}, {cnt} edges (expected {n_edges})")
        launches_per_step = 2   # hash insert and covers (after a memset of the table)
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier(world)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ms, kms = [], []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    for _ in range(args.steps):
        flush.zero_()
        ev0.record(stream)
        step()
        ev1.record(stream)
        ev1.synchronize()
        ms.append(ev0.elapsed_time(ev1))
        kms.append(ctx.stats()["lattice_ms"])   # the library's own events around its kernels
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    total_s = max_over_ranks(sum(ms) / 1e3, world)
    value = k * args.steps * world / total_s
    peaks = load_peaks() or {}
    result = {
        "metric": f"{args.stage}_concepts_per_s", "value": value, "unit": "concepts/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": w.name, "n_objects": w.n_objects, "n_attrs": w.n_attrs, "seed": w.seed,
                   "concepts": k, "stage": args.stage, "l2": "flushed between timed steps (512 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    mean_ms = statistics.mean(kms)
    result["kernel_ms_per_step"] = {("extents_kernel" if args.stage == "extents" else "covers"): mean_ms}
    if args.stage == "extents":
        # algorithmic bytes: intents read, extents written, the columns read once
        alg = k * (wm + wn) * 4 + w.n_attrs * ((wn + 3) // 4 * 4) * 4
        peak = peaks.get("hbm_gbs")
        achieved = alg / (mean_ms * 1e-3) / 1e9
        # DRAM bytes per launch from the committed ncu summary (captured on the workload's first rows;
        # the traffic grows with the rows, so it is scaled to this launch's rows)
        per_row = profile_traffic_per_row("extents_kernel", w.name)
        result["roofline"] = {"kernel": "extents_kernel", "bound": "hbm", "achieved": achieved,
                              "peak": peak, "unit": "GB/s", "frac": achieved / peak if peak else None,
                              "traffic": per_row * k if per_row is not None else None, "algorithmic_bytes": alg,
                              "basis": "library events around the one launch; peak: measured copy bandwidth"}
    else:
        result["edges"] = n_edges
        result["edges_per_s"] = n_edges * args.steps * world / total_s
        # algorithmic work of the lower-cover search over the whole intent set (oracle/coverwork.c,
        # stored by tests/golden/make_work_counts.py --covers): per concept its extent, the
        # intersections A & column k for k outside B, the closure of each non-empty one by rows
        cw = load_cover_counts(w.name)
        if cw is not None and cw.get("concepts") == k:
            sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
            sm_max = float(peaks.get("sm_max_mhz", 2070.0))
            probes = probe_peaks() if rank == 0 else {}
            hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
            hbm_basis = "MEASURED_PEAKS.json hbm_gbs" if "hbm_gbs" in peaks else "fallback 6.8 TB/s"
            l2_peak = probes.get("l2_read_gbs") or hbm_peak
            int_peak = sm_count * INT_LANES_PER_SM * sm_max * 1e6 / 1e9
            ops = cw["extent_words"] + cw["isect_words"] + cw["closure_words"]
            hbm_b = 4.0 * k * wm + 8.0 * n_edges                 # intents read, edges written
            l2_b = 4.0 * (cw["isect_words"] + cw["closure_words"])   # column and row words
            r = bound_of(hbm_b, l2_b, ops, 1, mean_ms, hbm_peak, hbm_basis, l2_peak, int_peak, sm_count, sm_max)
            result["roofline"] = {"kernel": "covers_kernel", **r,
                                  "traffic": profile_traffic("covers_kernel", w.name),
                                  "basis": "algorithmic work of the lower-cover search (oracle/coverwork.c); "
                                           "time: library events around the hash-insert and covers launches"}
        else:
            result["roofline"] = None
            result["roofline_note"] = "no stored cover-search work counts for this workload"
    ctx.close()
    return result


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as the reference arm: same workload, metric and unit, on the host cores.

    Each step is one bounded sample of the workload (the budget split over the steps, so the
    whole run stays within a few minutes)."""
    w = cx.WORKLOADS[args.workload]
    rows = w.rows()
    threads = os.cpu_count() or 1
    sampler = OracleSampler(rows, w, threads)
    per_step = max(0.5, min(args.cpu_seconds * 6, 120.0) / max(1, args.steps))
    for _ in range(max(args.warmup, 0)):
        sampler.sample(min(per_step, 1.0))
    rates, samples, seconds = [], [], 0.0
    for _ in range(max(1, args.steps)):
        rate, sample, dt = sampler.sample(per_step)
        rates.append(rate)
        samples.append(sample)
        seconds += dt
    value = statistics.median(rates)
    cb = {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": samples[-1],
          "seconds": round(seconds, 2)}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": len(rates), "warmup": args.warmup, "ms_per_step": seconds * 1e3 / len(rates),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u64",
            "data": "synthetic",
            "config": {"workload": w.name, "n_objects": w.n_objects, "n_attrs": w.n_attrs, "seed": w.seed},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.stage != "enumerate":
        result = run_lattice(args, world, rank, local)
        if rank == 0:
            print(json.dumps(result), flush=True)
        return
    result = run_ours(args, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            w = cx.WORKLOADS[args.workload]
            result["cpu_baseline"] = cpu_baseline(w.rows(), w, args.cpu_seconds)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
