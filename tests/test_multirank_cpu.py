"""Host-side logic of multi-rank benchmark runs, on CPU with the gloo backend.

The library itself runs on one GPU; under torchrun the benchmark runs one
independent replica per rank (no data-path collective) and combines the
per-rank numbers with a max (time) and a sum (work). These tests exercise
that combination and the rank-0-only reference arm with two CPU ranks.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        t_max = bench.reduce_max(0.5 + rank, "cpu")      # per-rank times
        units = bench.reduce_sum(10.0 * (rank + 1), "cpu")  # per-rank work
        out_q.put((rank, t_max, units))
    finally:
        dist.destroy_process_group()


def test_rank_time_max_and_work_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time and the total work of both
    assert results == [(0, 1.5, 30.0), (1, 1.5, 30.0)]


def test_helpers_are_identity_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert not dist.is_initialized()
    assert bench.reduce_max(2.5, "cpu") == 2.5
    assert bench.reduce_sum(4.0, "cpu") == 4.0
    bench.barrier()


def test_reference_arm_prints_one_line_from_rank_zero_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
