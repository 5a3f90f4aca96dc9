"""The benchmark's multi-rank host logic on CPU: two gloo ranks agree on the slowest
rank's numbers, whole-job throughput counts every rank's rows, and a two-rank torchrun
launch of the reference arm prints exactly one line (rank 0) and exits 0 on every rank.

Rows are independent, so several GPUs run replicas (weak scaling) with no collective on
the data path; the only cross-rank step is this timing reduction."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], "cpu")
        out_q.put((rank, vals))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(q.get() for _ in range(2))
    assert got[0] == got[1] == [2.0, 10.0, 3.5]


def test_single_process_values_pass_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 256 rows x 10 steps over the slowest rank's 20 ms
    assert bench.job_rows_per_s(2, 256, 10, 20.0) == pytest.approx(256000.0)
    assert bench.job_rows_per_s(1, 256, 1, 0.5) == pytest.approx(512000.0)


def test_reference_arm_under_a_two_rank_launch():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-rows", "2", "--workload", "small_mixed"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "rows/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
