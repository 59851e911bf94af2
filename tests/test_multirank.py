"""The multi-rank host path of bench.py on the CPU (gloo, world size 2).

Every box here has one GPU, so `bench.py --gpus N` runs N independent replicas: no collective on the
data path, only the timing barrier and the maximum of the ranks' times. These tests run that host
logic as two gloo ranks: the process-group set-up from the launcher's environment, the barrier, the
max-over-ranks reduction, and the reference arm under the launcher (rank 0 alone prints its line).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    got = bench.max_over_ranks(1.5 + rank, w)     # each rank's elapsed time; the job's is the largest
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time(tmp_path):
    port = free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        assert json.load(open(tmp_path / f"rank{rank}.json"))["max"] == 2.5


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_setup(1) == (1, 0, 0)
        assert bench.max_over_ranks(3.25, 1) == 3.25
        bench.barrier(1)
    finally:
        os.environ.update(env)


def test_reference_arm_under_the_launcher_prints_once():
    """`torchrun --nproc-per-node 2 bench.py --impl reference`: rank 0 times the oracle and prints one
    JSON line; rank 1 exits 0 without work."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "1",
           "--cpu-seconds", "0.2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
