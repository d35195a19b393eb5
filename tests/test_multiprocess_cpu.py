"""The benchmark's multi-process path on the CPU (gloo, world size 2, 127.0.0.1).

Sequences are independent: rank r takes its share of a global batch of (world x 32) sequences, each
drawn from its own seeds; the only cross-rank operations are a barrier, the max of the per-rank step
times and the sum of the ranks' token counts (no data-path collective).  These tests run that
plumbing with the gloo backend, and check that a batch computed in shards (by the oracle: no GPU is
involved) equals the same batch computed by one rank.
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


def _shard_main(rank, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    from linear_attention_kda_gb300 import synthetic as syn
    from oracle import numpy_ref as NR
    r, ws, _ = bench.dist_setup()
    w = syn.Workload("shard_tiny", H=2, d=16, dtype="f32", n_seq=3, seq_len=None, len_lo=1, len_hi=150,
                     z_std=1.5, b_range=1.0, alog_std=0.25, s0_std=0.02)
    d = syn.make_prefill_shard(w, 11, r, ws)
    o, st = NR.forward(d["q"], d["k"], d["v"], d["z"], d["beta"], d["dt_bias"], d["A_log"], d["cu_seqlens"],
                       S0=d["initial_state"])
    cu = [int(x) for x in d["cu_seqlens"]]
    mine = {i: (o[cu[j]:cu[j + 1]], st[j]) for j, i in enumerate(d["seq_ids"])}
    total = bench.sum_over_ranks(float(cu[-1]), ws)
    got = [None] * ws if r == 0 else None
    dist.gather_object(mine, got, dst=0)
    if r == 0:
        q.put(({k: v for part in got for k, v in part.items()}, total))
    dist.destroy_process_group()


def test_sharded_batch_equals_one_rank():
    """Two gloo ranks each compute their shard of a 6-sequence batch (ragged lengths 1..150, states);
    the union of the shards' outputs and final states equals the whole batch computed by one rank,
    every sequence is computed exactly once, and the token count summed over ranks is the batch's."""
    import numpy as np
    from linear_attention_kda_gb300 import synthetic as syn
    from oracle import numpy_ref as NR
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    shards, total = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w1 = syn.Workload("shard_tiny", H=2, d=16, dtype="f32", n_seq=6, seq_len=None, len_lo=1, len_hi=150,
                      z_std=1.5, b_range=1.0, alog_std=0.25, s0_std=0.02)
    d = syn.make_prefill_shard(w1, 11, 0, 1)
    o, st = NR.forward(d["q"], d["k"], d["v"], d["z"], d["beta"], d["dt_bias"], d["A_log"], d["cu_seqlens"],
                       S0=d["initial_state"])
    cu = [int(x) for x in d["cu_seqlens"]]
    assert sorted(shards) == list(range(6)) and total == cu[-1]
    for j in range(6):
        os_, ss_ = shards[j]
        assert np.array_equal(os_, o[cu[j]:cu[j + 1]]) and np.array_equal(ss_, st[j])


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
