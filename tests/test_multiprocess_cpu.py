"""The benchmark's multi-process path on the CPU (gloo, world size 2, 127.0.0.1).

The path shards by replicas: every rank runs the same workload, the only cross-rank operations are
a barrier and the max of the per-rank step times (no data-path collective).  These tests run that
plumbing with the gloo backend; no GPU is involved.
"""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, ws, local = bench.dist_setup()
    bench.barrier(ws)
    worst = bench.max_over_ranks(10.0 + 5.0 * r, ws)  # rank 1 is the slower one
    q.put((r, ws, local, worst, dist.get_backend()))
    dist.destroy_process_group()


def test_dist_helpers_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    for r, ws, local, worst, backend in res:
        assert ws == 2 and local == r and backend == "gloo"
        assert worst == 15.0  # every rank reports the slowest rank's time


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` under torchrun with 2 ranks: rank 0 alone runs the oracle and
    prints one JSON line; the other rank exits 0 without work."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="4")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
