"""The multi-rank host logic of bench.py on CPU: replicas reduce their step time to the
slowest rank's (gloo, world size 2), and the reference arm under torchrun prints one line
from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [0.40, 0.55][rank]  # rank 1 is the slow one
        worst = bench.max_over_ranks(ms, dist, "cpu")
        q.put((rank, worst, bench.job_throughput(1.0e12, worst, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [0.55, 0.55]
    # both ranks' work (2 x 1 TFLOP) over the slowest rank's 0.55 ms
    assert all(abs(o[2] - 2.0 / 0.55e-3) < 1e-6 for o in out)


def test_single_process_helpers():
    assert bench.max_over_ranks(0.7) == 0.7
    assert abs(bench.job_throughput(0.55e12, 0.5, 1) - 1100.0) < 1e-9


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1",
           "--warmup", "3", "--ref-step-seconds", "0.05"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
