"""KDA benchmark: chunked prefill (tokens/s, TFLOP/s) and decode (GB/s) on one GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one kda_chunk_fwd pass over the varlen bf16 prefill batch (32
sequences with lengths uniform in [512, 8192], ~140K tokens packed by
cu_seqlens, H=32, d_k=d_v=128, C=64, fp32 initial states in and final states
out), inputs resident in HBM.  L2 is flushed (a 512 MiB write) before every
timed step (the step's inputs, ~180 MB, also exceed L2); each step is timed
alone with CUDA events on the launching stream, and per-kernel times come from
events the library records between its launches.  The single-sequence T=4096
prefill (a latency figure: one 64-chunk chain per head), the 1M-token
sequence, the output epilogue, the softplus gate, the backward pass and the
decode workload (256 sequences x 32 heads, 512 in-place steps) are measured in
the same run.  Under torchrun each rank runs its own copy of the workload
(sequences are independent: no data-path collective); value = tokens of all
ranks / max time over ranks.

--impl reference times the fp64 CPU oracle (test infrastructure) on a bounded
sample of the same workload, on the host cores, as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_attention_kda_gb300 import synthetic as syn  # noqa: E402

METRIC = "KDA chunked prefill tokens/s and TFLOP/s (% BF16 TC peak); decode GB/s (% HBM)"
WORKLOAD = syn.VARLEN_32     # headline: the varlen batch, T >= 64K tokens
LATENCY = syn.PREFILL_4K     # one 4096-token sequence: latency-bound (a 64-step chain per head)
LONG = syn.LONG_1M           # one 1M-token sequence
DECODE = syn.DECODE_256
ORACLE_SAMPLE_UNITS = 48     # (sequence, head) units of the varlen batch per oracle step
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- accounting

def chunk_lengths(lengths, C):
    out = []
    for L in lengths:
        full, tail = divmod(int(L), C)
        out += [C] * full + ([tail] if tail else [])
    return out


def prefill_flops(lengths, H, dk, dv, C=64):
    """Algorithmic FLOPs (2 per MAC, causal shapes) of the chunked form, split by kernel role.

    intra (UT transform, A):  2 dk c(c+1) + dk c(c-1) + dv c(c+1) + c^3/3
    inter (state, output):    6 c dk dv + dv c(c+1)
    """
    intra = inter = dense = 0.0
    for c in chunk_lengths(lengths, C):
        intra += 2 * dk * c * (c + 1) + dk * c * (c - 1) + dv * c * (c + 1) + c ** 3 / 3.0
        inter += 6 * c * dk * dv + dv * c * (c + 1)
        dense += 6 * C * dk * dv + 3 * (2 * C * C * dk) + 2 * (2 * C * C * dv) + C ** 3 / 3.0
    return {"intra": intra * H, "inter": inter * H, "total": (intra + inter) * H, "dense_tile": dense * H}


def prefill_bytes(T, N, H, dk, dv, io_bytes, with_s0, with_sT):
    """Algorithmic HBM bytes: read q, k, z [dk], v [dv], beta; write o [dv]; states fp32."""
    per_tok_in = (3 * dk + dv) * io_bytes + io_bytes
    per_tok_out = dv * io_bytes
    st = N * H * dk * dv * 4
    return {"intra": T * H * per_tok_in,
            "inter": T * H * per_tok_out + (st if with_s0 else 0) + (st if with_sT else 0),
            "total": T * H * (per_tok_in + per_tok_out) + (st if with_s0 else 0) + (st if with_sT else 0)}


def decode_bytes(N, H, d, io_bytes):
    """Per step: state read + write (fp32), q, k, v, z, beta read, o written."""
    return N * H * (2 * d * d * 4 + 4 * d * io_bytes + io_bytes + d * io_bytes)


def chunk_lengths_count(lengths, C=64):
    return [(int(L) + C - 1) // C for L in lengths]


def kernel_names(sch, nk):
    """Names of the kernels kda_chunk_fwd launches under schedule `sch` (kda_chunk_fwd_schedule)."""
    if sch.get("team"):
        return ["chunk_team"] + ["output_gate"] * (nk - 1)
    if sch["fused"]:
        return ["chunk_fused"] + ["output_gate"] * (nk - 1)
    base = ["chunk_plan", "chunk_intra"] + (["chunk_segsum", "chunk_fold"] if sch["seg_len"] else []) + ["chunk_inter"]
    return base + ["output_gate"] * (nk - len(base))


def schedule_name(sch):
    if sch.get("team"):
        return "chain teams (1 chain CTA + %d producer CTAs each, producers a bounded window ahead)" % sch["team_producers"]
    if sch["fused"]:
        return "fused"
    return "split state pass, %d chunks per segment" % sch["seg_len"] if sch["seg_len"] else "separate kernels"


def timed_steps(fn, flush, stream, warmup, steps):
    """Mean CUDA-event time (ms) of `steps` calls of fn, each after an L2 flush, after `warmup` calls."""
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(steps):
        flush.zero_()
        ea.record(stream)
        fn()
        eb.record(stream)
        eb.synchronize()
        ts.append(ea.elapsed_time(eb))
    return sum(ts) / len(ts)


def measured_traffic(kernel, p_items):
    """DRAM bytes per launch of `kernel` from the committed ncu record (profiles/traffic_*.json),
    scaled by the work items of this launch (the record's unit: (chunk, head) items of the prefill,
    (sequence, head) states of the replay window); None if no record exists or the kernel source
    changed since the capture (sha256 prefix mismatch)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != rec["source_sha256_16"]:
            return None
    return rec["dram_bytes_per_item"] * p_items


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock, power and clock-event reasons during the timed region (read-only).

    Uses NVML through ctypes every 2 ms (the timed regions are tens of milliseconds); falls back
    to `nvidia-smi -lms 100` when NVML cannot be loaded.  Nothing here changes any GPU setting.
    """

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index=0, period_s=0.002):
        self.index = index
        self.period = period_s
        self.rows = []
        self.proc = None
        self.nvml = None
        self.thread = None
        self.stop = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return None
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return lib, h, reasons

    def _poll(self):
        import ctypes
        lib, h, reasons = self.nvml
        clk, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        while not self.stop.is_set():
            lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))  # NVML_CLOCK_SM
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            reasons(h, ctypes.byref(rs))
            self.rows.append((float(clk.value), float(mx.value), pw.value / 1000.0, int(rs.value)))
            time.sleep(self.period)

    def __enter__(self):
        import threading
        try:
            self.nvml = self._nvml_open()
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        self.path = os.path.join("/tmp", f"kda_clocks_{os.getpid()}.csv")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
            with open(self.path) as f:
                for ln in f:
                    parts = [x.strip() for x in ln.split(",")]
                    try:
                        self.rows.append((float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3], 16)))
                    except (ValueError, IndexError):
                        continue

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"]}
        reasons = sorted({name for r in self.rows for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[0] for r in self.rows), "sm_max_mhz": max(r[1] for r in self.rows),
                "power_w_max": max(r[2] for r in self.rows), "samples": len(self.rows),
                "source": "nvml" if self.nvml is not None else "nvidia-smi", "reasons": reasons}


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def sum_over_ranks(x, ws):
    """Sum of a per-rank host value (token counts of the ranks' shards)."""
    if ws <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def max_over_ranks(x, ws):
    if ws <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle

def cpu_oracle_run(d, units=None, reps_target_s=10.0, max_reps=3):
    """Times the fp64 C oracle (as it stands) on the workload; returns (token-heads/s, threads, secs)."""
    from oracle import c_ref
    c_ref.build()
    nth = os.cpu_count() or 1
    best = None
    used = 1
    total = 0.0
    reps = 0
    while reps < max_reps and (reps == 0 or total < reps_target_s):
        _, info = c_ref.forward(d["q"], d["k"], d["v"], d["z"], d["beta"], d["dt_bias"], d["A_log"],
                                d["cu_seqlens"], S0=d["initial_state"], units=units, nthreads=nth)
        used = info["threads"]
        total += info["seconds"]
        best = info["seconds"] if best is None else min(best, info["seconds"])
        reps += 1
    return best, used, total, reps


def workload_config(w, lengths, ws):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": w.name, "tokens": int(sum(lengths)), "sequences": len(lengths), "heads": w.H,
            "d_k": w.d, "d_v": w.d, "chunk": 64, "io_dtype": w.dtype, "state_dtype": "f32",
            "initial_state": w.s0_std > 0, "final_state": True,
            "l2": "flushed (512 MiB write) before every timed step; inputs exceed L2",
            "parallelism": f"sequence shards x{ws}" if ws > 1 else "one GPU",
            "global_sequences": len(lengths) * ws, "tokens_per_rank": int(sum(lengths))}


def oracle_sample_units(lengths, H, n_units=ORACLE_SAMPLE_UNITS, seed=5):
    """A seeded sample of (sequence, head) units of the workload for the CPU oracle."""
    g = torch.Generator().manual_seed(seed)
    pick = torch.randperm(len(lengths) * H, generator=g)[:n_units].tolist()
    units = [(i // H, i % H) for i in pick]
    return units, sum(int(lengths[n]) for n, _ in units)


def run_reference(args, rank, ws):
    if rank != 0:
        return
    d = syn.make_prefill_shard(WORKLOAD, 2, 0, 1, device="cpu")
    lengths = d["lengths"]
    H = WORKLOAD.H
    units, th = oracle_sample_units(lengths, H)
    from oracle import c_ref
    c_ref.build()
    nth = os.cpu_count() or 1
    times = []
    used = 1
    for i in range(args.warmup + args.steps):
        _, info = c_ref.forward(d["q"], d["k"], d["v"], d["z"], d["beta"], d["dt_bias"], d["A_log"],
                                d["cu_seqlens"], S0=d["initial_state"], units=units, nthreads=nth)
        used = info["threads"]
        if i >= args.warmup:
            times.append(info["seconds"])
    secs = sum(times) / len(times)
    value = th / H / secs  # token-heads/s of the sample, in tokens (of all H heads) per second
    ms = 1e3 * sum(lengths) / value  # time the oracle would take for one whole step at that rate
    sample = (f"{len(units)} seeded (sequence, head) units of the batch ({th} token-heads) per step; "
              f"value = sampled token-heads/s / {H} heads")
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(WORKLOAD, lengths, ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args, rank, ws, local):
    from linear_attention_kda_gb300 import build as kbuild, kda
    kbuild.build()
    kda.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    stream = torch.cuda.current_stream(dev)

    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tc = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    flush = torch.empty((512 << 20,), dtype=torch.uint8, device=dev)

    # ---------------- headline: the varlen batch, inputs resident in HBM
    # rank r's shard of a global batch of ws x 32 sequences (each sequence drawn from its own seeds, so
    # it is the same whatever the number of ranks): weak scaling, no data-path collective
    d = syn.make_prefill_shard(WORKLOAD, 2, rank, ws, device=dev)
    lengths = d["lengths"]
    T, N, H, D = sum(lengths), len(lengths), WORKLOAD.H, WORKLOAD.d
    cu_host = d["cu_seqlens"].cpu()
    q, k, v, z, beta = (d[n] for n in ("q", "k", "v", "z", "beta"))
    b, a, s0 = d["dt_bias"], d["A_log"], d["initial_state"]
    o = torch.empty_like(v)
    fs = torch.empty((N, H, D, D), dtype=torch.float32, device=dev)
    wsz = kda.chunk_fwd_workspace_size(T, N, H, D, D, q.dtype, 64, cu_host)
    work = torch.empty((wsz,), dtype=torch.uint8, device=dev)

    def step():
        kda.chunk_fwd(q, k, v, z, beta, b, a, g_min=d["g_min"], scale=d["scale"], cu_seqlens=d["cu_seqlens"],
                      cu_seqlens_host=cu_host, initial_state=s0, final_state=fs, workspace=work, out=o)

    nk = kda.chunk_fwd_kernel_count(T, N, H, D, D, q.dtype, cu_host)
    sch = kda.chunk_fwd_schedule(T, N, H, D, D, q.dtype, cu_host)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    for row in ev:  # materialise the events before handing them to the library
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(ws)
        # headline: whole steps, nothing recorded between the library's launches
        for i in range(args.steps):
            flush.zero_()
            ev_step[i][0].record(stream)
            step()
            ev_step[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        # per-kernel breakdown: the same steps with the library's events recorded between its launches
        for i in range(args.steps):
            flush.zero_()
            kda.set_profile_events(ev[i])
            step()
        kda.set_profile_events([])
        torch.cuda.synchronize()
        barrier(ws)
    clocks = clk.summary()
    step_ms = [ev_step[i][0].elapsed_time(ev_step[i][1]) for i in range(args.steps)]
    step_ms_marked = [ev[i][0].elapsed_time(ev[i][nk]) for i in range(args.steps)]
    kern_ms = [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)] for j in range(nk)]
    ms = sum(step_ms) / len(step_ms)
    step_spread = [min(step_ms), sorted(step_ms)[len(step_ms) // 2], max(step_ms)]
    ms_max = max_over_ranks(ms, ws)
    T_all = sum_over_ranks(float(T), ws)  # tokens of every rank's shard
    value = T_all / (ms_max / 1e3)
    fl = prefill_flops(lengths, H, D, D)
    by = prefill_bytes(T, N, H, D, D, 2, s0 is not None, True)
    tflops = fl["total"] / (ms / 1e3) / 1e12
    kern_avg = [sum(x) / len(x) for x in kern_ms]
    names = kernel_names(sch, nk)
    dom = max(range(nk), key=lambda j: kern_avg[j])
    role = {"chunk_intra": "intra", "chunk_fused": "total", "chunk_team": "total"}.get(names[dom], "inter")
    bytes_dom, flops_dom = by[role], fl[role]
    t_dom = kern_avg[dom] / 1e3
    # the kernel's algorithmic bound: whichever of its bytes or FLOPs takes longer at peak
    if bytes_dom / (hbm * 1e9) >= flops_dom / (tc * 1e12):
        roof = {"bound": "hbm", "achieved": bytes_dom / t_dom / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops_dom / t_dom / 1e12, "peak": tc, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(names[dom], p_items=sum(chunk_lengths_count(lengths)) * H)
    roof["kernel"] = names[dom]
    roof["algorithmic_bytes"] = bytes_dom
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json burst)" if peak_kind == "measured" else "fallback"

    # ---------------- e2e through the same C ABI call with host buffers
    in_names = ("q", "k", "v", "z", "beta", "initial_state")
    pin = {n: d[n].cpu().pin_memory() for n in in_names}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    fs_host = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = o_host.numel() * o_host.element_size() + fs_host.numel() * fs_host.element_size()

    def run_on(di, o_, fs_):
        kda.chunk_fwd(di["q"], di["k"], di["v"], di["z"], di["beta"], b, a, g_min=d["g_min"], scale=d["scale"],
                      cu_seqlens=d["cu_seqlens"], cu_seqlens_host=cu_host, initial_state=di["initial_state"],
                      final_state=fs_, workspace=work, out=o_)

    dev_in = {n: torch.empty_like(d[n]) for n in pin}

    def e2e_step():
        for n in pin:
            dev_in[n].copy_(pin[n], non_blocking=True)
        run_on(dev_in, o, fs)
        o_host.copy_(o, non_blocking=True)
        fs_host.copy_(fs, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_times = []
    barrier(ws)
    for _ in range(args.steps):
        flush.zero_()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_times.append(e0.elapsed_time(e1))
    e2e_ms = max_over_ranks(sum(e2e_times) / len(e2e_times), ws)

    # pipelined: two device buffers for inputs and results; step s + 1's inputs cross the link on a
    # copy stream while step s computes, step s's results return on a third stream.  Every step's
    # inputs are still copied from pinned host memory and every step's result read back, inside the
    # timed region (from the first copy issued to the last result landed).
    dev_in2 = [dev_in, {n: torch.empty_like(d[n]) for n in pin}]
    o2_ = [o, torch.empty_like(o)]
    fs2_ = [fs, torch.empty_like(fs)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_back = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(sidx):
        bi = sidx & 1
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(ev_done[bi])  # the step that last used this buffer has computed
            for n in pin:
                dev_in2[bi][n].copy_(pin[n], non_blocking=True)
            ev_in[bi].record(s_h2d)

    def pipelined(nsteps):
        for e_ in ev_done + ev_back:
            e_.record(stream)
        copy_in(0)
        for sidx in range(nsteps):
            bi = sidx & 1
            if sidx + 1 < nsteps:
                copy_in(sidx + 1)
            stream.wait_event(ev_in[bi])
            stream.wait_event(ev_back[bi])  # this result buffer has been read back
            run_on(dev_in2[bi], o2_[bi], fs2_[bi])
            ev_done[bi].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[bi])
                o_host.copy_(o2_[bi], non_blocking=True)
                fs_host.copy_(fs2_[bi], non_blocking=True)
                ev_back[bi].record(s_d2h)

    pipelined(args.warmup)
    torch.cuda.synchronize()
    barrier(ws)
    t0_ = time.perf_counter()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(s_h2d)
    pipelined(args.steps)
    p1.record(s_d2h)  # after the last read-back, which waits on the last step's compute
    p1.synchronize()
    e2e_pipe_ms = max_over_ranks(p0.elapsed_time(p1) / args.steps, ws)
    e2e_pipe_wall_ms = (time.perf_counter() - t0_) * 1e3 / args.steps
    del dev_in, dev_in2, pin, o2_, fs2_
    T_head, ms_head = T, ms

    del q, k, v, z, beta, d, o, fs, work
    torch.cuda.empty_cache()

    # ---------------- latency figure: one 4096-token sequence (a 64-step chain per head)
    d = syn.make_prefill(LATENCY, seed=1 + rank, device=dev)
    lengths4 = d["lengths"]
    T4 = sum(lengths4)
    cu_host4 = d["cu_seqlens"].cpu()
    q, k, v, z, beta = (d[n] for n in ("q", "k", "v", "z", "beta"))
    b, a = d["dt_bias"], d["A_log"]
    o = torch.empty_like(v)
    fs = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
    work = torch.empty((kda.chunk_fwd_workspace_size(T4, 1, H, D, D, q.dtype, 64, cu_host4),), dtype=torch.uint8,
                       device=dev)

    def step4():
        kda.chunk_fwd(q, k, v, z, beta, b, a, g_min=d["g_min"], scale=d["scale"], cu_seqlens=d["cu_seqlens"],
                      cu_seqlens_host=cu_host4, final_state=fs, workspace=work, out=o)

    ms4 = timed_steps(step4, flush, stream, args.warmup, args.steps)
    fl4 = prefill_flops(lengths4, H, D, D)
    by4 = prefill_bytes(T4, 1, H, D, D, 2, False, True)
    sch4 = kda.chunk_fwd_schedule(T4, 1, H, D, D, q.dtype, cu_host4)
    lat = {"workload": LATENCY.name, "tokens": T4, "ms_per_step": ms4, "tokens_per_s": T4 / (ms4 / 1e3),
           "tflops": fl4["total"] / (ms4 / 1e3) / 1e12, "frac_bf16_peak": fl4["total"] / (ms4 / 1e3) / 1e12 / tc,
           "frac_hbm": by4["total"] / (ms4 / 1e3) / 1e9 / hbm, "schedule": schedule_name(sch4),
           "l2": "flushed (512 MiB write) before every timed step"}
    ms = ms4  # the side measurements below (epilogue, softplus gate, backward) run on this workload
    T, N = T4, 1
    cu_host = cu_host4
    fs = fs[:1]

    # ---------------- output epilogue of Eq. 6: through kda_chunk_fwd, and the pass alone
    epi = None
    if not args.no_epilogue:
        g_in, w_in = syn.make_output_gate_inputs(T, H, D, "bf16", 33 + rank, device=dev)
        o2 = torch.empty_like(v)

        def step_epi():
            kda.chunk_fwd(q, k, v, z, beta, b, a, g_min=d["g_min"], scale=d["scale"], cu_seqlens=d["cu_seqlens"],
                          cu_seqlens_host=cu_host, final_state=fs, workspace=work, out=o2, out_gate=g_in,
                          out_norm_weight=w_in, out_norm_eps=1e-6)

        def sep_pass():
            kda.output_gate(o, g_in, w_in, 1e-6, out=o2)

        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def timed(fn, n):
            ts = []
            for _ in range(n):
                flush.zero_()
                ea.record(stream)
                fn()
                eb.record(stream)
                eb.synchronize()
                ts.append(ea.elapsed_time(eb))
            return sum(ts) / len(ts)

        for _ in range(3):
            flush.zero_()
            step_epi()
            sep_pass()
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        ms_fused = timed(step_epi, args.steps)
        ms_sep = timed(sep_pass, args.steps)
        ob = 3 * T * H * D * 2 + H * D * 4  # o and g read, y written (bf16), weight
        gb = ob / (ms_sep / 1e3) / 1e9
        del g_in, w_in, o2
        # the pass alone at the headline batch's size (138,111 tokens x 32 heads: 3.4 GB moved), where the
        # launch and the first misses after the L2 flush no longer dominate (at T = 4096 they are ~1/3)
        Tb = int(T_head)
        ob_big = torch.randn(Tb, H, D, device=dev).to(torch.bfloat16)
        g_big, w_big = syn.make_output_gate_inputs(Tb, H, D, "bf16", 34 + rank, device=dev)
        y_big = torch.empty_like(ob_big)
        for _ in range(3):
            kda.output_gate(ob_big, g_big, w_big, 1e-6, out=y_big)
        ms_big = timed(lambda: kda.output_gate(ob_big, g_big, w_big, 1e-6, out=y_big), max(5, args.steps // 4))
        bytes_big = 3 * Tb * H * D * 2 + H * D * 4
        gb_big = bytes_big / (ms_big / 1e3) / 1e9
        del ob_big, g_big, w_big, y_big
        epi = {"what": "o <- Sigmoid(g) * RMSNorm(o) per (token, head) (Eq. 6 without projections)",
               "prefill_with_epilogue_ms_per_step": ms_fused, "epilogue_overhead_ms": ms_fused - ms,
               "epilogue_pass_ms": ms_sep,
               "pass_at_T4096": {"GB_per_s": gb, "frac": gb / hbm, "bytes": ob},
               "roofline": {"bound": "hbm", "achieved": gb_big, "peak": hbm, "unit": "GB/s",
                            "frac": gb_big / hbm, "bytes": bytes_big, "kernel": "output_gate",
                            "workload": f"output_gate_bf16_T{Tb}_H{H}_d{D}", "ms": ms_big}}

    # ---------------- what the bounded gate buys (section 2.1.1): the same prefill with the unbounded
    # softplus gate, which has to take the fp32 CUDA-core path (its in-chunk decays are not bounded)
    gvar = None
    if not args.no_gate_variant:
        need_sp = kda.chunk_fwd_workspace_size(T, N, H, D, D, q.dtype, 64, cu_host, gate="softplus")
        work_sp = torch.empty((need_sp,), dtype=torch.uint8, device=dev)
        o_sp, fs_sp = torch.empty_like(v), torch.empty_like(fs)

        def step_sp():
            kda.chunk_fwd(q, k, v, z, beta, b, a, scale=d["scale"], cu_seqlens=d["cu_seqlens"],
                          cu_seqlens_host=cu_host, final_state=fs_sp, workspace=work_sp, out=o_sp, gate="softplus")

        for _ in range(3):
            flush.zero_()
            step_sp()
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        sa, sb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sp_ts = []
        for _ in range(max(3, min(args.steps, 10))):
            flush.zero_()
            sa.record(stream)
            step_sp()
            sb.record(stream)
            sb.synchronize()
            sp_ts.append(sa.elapsed_time(sb))
        ms_sp = sum(sp_ts) / len(sp_ts)
        gvar = {"what": "the same step with g = -exp(A) Softplus(z + b) (unbounded): fp32 CUDA-core path",
                "softplus_ms_per_step": ms_sp, "lower_bound_ms_per_step": ms,
                "softplus_tokens_per_s": T / (ms_sp / 1e3), "slowdown": ms_sp / ms,
                "kernels": kda.chunk_fwd_kernel_count(T, N, H, D, D, q.dtype, cu_host, gate="softplus")}
        del work_sp, o_sp, fs_sp

    # ---------------- backward pass (training) on the same workload: gradients of q, k, v, z, beta, dt_bias,
    # A_log from grad_o and grad_final_state (the forward recomputed inside; chains and value side on the
    # tensor cores for this bf16 d = 128 workload)
    bwd = None
    if not args.no_backward:
        gen = torch.Generator(device=dev).manual_seed(77 + rank)
        go = torch.randn(o.shape, generator=gen, device=dev).to(o.dtype)
        gST = torch.randn(fs.shape, generator=gen, device=dev) * 0.1
        need_b = kda.load_library().kda_chunk_bwd_workspace_size(T, N, H, D, D, 64)
        work_b = torch.empty((need_b,), dtype=torch.uint8, device=dev)

        def step_b():
            return kda.chunk_bwd(q, k, v, z, beta, b, a, go, g_min=d["g_min"], scale=d["scale"],
                                 cu_seqlens=d["cu_seqlens"], grad_final_state=gST, workspace=work_b)

        for _ in range(2):
            flush.zero_()
            step_b()
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        nb = 8  # plan, intra, forward chain with checkpoints, reverse chain, value side, key side, gate params
        evb = [[torch.cuda.Event(enable_timing=True) for _ in range(nb)] for _ in range(max(3, min(args.steps, 10)))]
        for row in evb:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        for row in evb:
            flush.zero_()
            kda.set_profile_events(row)
            step_b()
        kda.set_profile_events([])
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        names_b = ["plan", "intra (fp32 records + L)", "forward chain (entering states)", "reverse chain",
                   "value side", "key side", "gate parameters"]
        per_b = [sum(r[i].elapsed_time(r[i + 1]) for r in evb) / len(evb) for i in range(nb - 1)]
        ms_b = sum(r[0].elapsed_time(r[nb - 1]) for r in evb) / len(evb)
        bwd = {"what": "kda_chunk_bwd: d q, k, v, z, beta, dt_bias, A_log, S0 from d o and d S_T",
               "ms_per_step": ms_b, "tokens_per_s": T / (ms_b / 1e3), "vs_forward": ms_b / ms,
               "kernels_ms": dict(zip(names_b, per_b)), "workspace_bytes": int(need_b)}
        del go, gST, work_b

    # ---------------- the long prefill workloads (T >= 64K): the varlen batch (32 sequences, ~140K tokens,
    # initial states) and the 1M-token sequence; inputs far exceed L2, so no flush is needed
    longw = None
    if not args.no_long:
        longw = {}
        for w_ in (LONG,):
            dl = syn.make_prefill(w_, seed=3, device=dev)
            Ls = dl["lengths"]
            Tl, Nl = sum(Ls), len(Ls)
            cul = dl["cu_seqlens"].cpu()
            fsl = torch.empty((Nl, H, D, D), dtype=torch.float32, device=dev)
            ol = torch.empty_like(dl["v"])
            wl = torch.empty((kda.chunk_fwd_workspace_size(Tl, Nl, H, D, D, dl["q"].dtype, 64, cul),),
                             dtype=torch.uint8, device=dev)

            def step_l():
                kda.chunk_fwd(dl["q"], dl["k"], dl["v"], dl["z"], dl["beta"], dl["dt_bias"], dl["A_log"],
                              cu_seqlens=dl["cu_seqlens"], cu_seqlens_host=cul, initial_state=dl["initial_state"],
                              final_state=fsl, workspace=wl, out=ol)

            for _ in range(2):
                step_l()
            torch.cuda.synchronize()
            assert kda.get_device_error() == 0
            la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            lts = []
            for _ in range(3):
                la.record(stream)
                step_l()
                lb.record(stream)
                lb.synchronize()
                lts.append(la.elapsed_time(lb))
            msl = sum(lts) / len(lts)
            epi_l = None
            if not args.no_epilogue:  # the same step with the Eq. 6 epilogue (applied inside the output pass)
                gl, wl_ = syn.make_output_gate_inputs(Tl, H, D, "bf16", 35, device=dev)

                def step_le():
                    kda.chunk_fwd(dl["q"], dl["k"], dl["v"], dl["z"], dl["beta"], dl["dt_bias"], dl["A_log"],
                                  cu_seqlens=dl["cu_seqlens"], cu_seqlens_host=cul,
                                  initial_state=dl["initial_state"], final_state=fsl, workspace=wl, out=ol,
                                  out_gate=gl, out_norm_weight=wl_, out_norm_eps=1e-6)

                step_le()
                torch.cuda.synchronize()
                assert kda.get_device_error() == 0
                ets = []
                for _ in range(3):
                    la.record(stream)
                    step_le()
                    lb.record(stream)
                    lb.synchronize()
                    ets.append(la.elapsed_time(lb))
                mse = sum(ets) / len(ets)
                epi_l = {"with_epilogue_ms_per_step": mse, "overhead": mse / msl - 1.0,
                         "kernels": kda.chunk_fwd_kernel_count(Tl, Nl, H, D, D, dl["q"].dtype, cul, out_gate=True)}
                del gl, wl_
            bwd_l = None
            if not args.no_backward and Nl == 1:
                # the backward of the whole sequence in a bounded workspace (32 GiB: segments of one
                # sequence; the one-pass scratch would be ~209 GiB)
                del wl
                torch.cuda.empty_cache()
                wl = None
                ws_b = 32 << 30
                full_b = kda.chunk_bwd_workspace_size(Tl, 1, H, D, D)
                wsb = torch.empty((min(ws_b, full_b),), dtype=torch.uint8, device=dev)
                gen = torch.Generator(device=dev).manual_seed(36)
                dol = torch.randn(ol.shape, generator=gen, device=dev).to(ol.dtype)

                def step_lb():
                    return kda.chunk_bwd(dl["q"], dl["k"], dl["v"], dl["z"], dl["beta"], dl["dt_bias"], dl["A_log"],
                                         dol, initial_state=dl["initial_state"], workspace=wsb)

                gb_ = step_lb()
                torch.cuda.synchronize()
                assert kda.get_device_error() == 0
                del gb_
                la.record(stream)
                gb_ = step_lb()
                lb.record(stream)
                lb.synchronize()
                msb = la.elapsed_time(lb)
                bwd_l = {"what": "kda_chunk_bwd of the whole sequence in a 32 GiB workspace (segments)",
                         "ms_per_step": msb, "tokens_per_s": Tl / (msb / 1e3), "vs_forward": msb / msl,
                         "workspace_bytes": int(wsb.numel()), "one_pass_workspace_bytes": int(full_b)}
                del gb_, wsb, dol
                torch.cuda.empty_cache()
            fll = prefill_flops(Ls, H, D, D)
            byl = prefill_bytes(Tl, Nl, H, D, D, 2, dl["initial_state"] is not None, True)
            tfl = fll["total"] / (msl / 1e3) / 1e12
            sch_l = kda.chunk_fwd_schedule(Tl, Nl, H, D, D, dl["q"].dtype, cul)
            longw[w_.name] = {
                "tokens": Tl, "sequences": Nl, "ms_per_step": msl, "tokens_per_s": Tl / (msl / 1e3),
                "tflops": tfl, "tflops_dense_tile": fll["dense_tile"] / (msl / 1e3) / 1e12,
                "frac_bf16_peak": tfl / tc, "hbm_gbs_algorithmic": byl["total"] / (msl / 1e3) / 1e9,
                "frac_hbm": byl["total"] / (msl / 1e3) / 1e9 / hbm,
                "schedule": schedule_name(sch_l), "kernels": sch_l["kernels"], "epilogue": epi_l,
                "backward": bwd_l}
            del dl, fsl, ol, wl
            torch.cuda.empty_cache()

    # ---------------- decode workload (HBM-bound), 512 in-place steps
    dec = None
    if not args.no_decode:
        dd = syn.make_decode(DECODE, seed=4 + rank, device=dev)
        st = dd["state"]
        nsteps = DECODE.decode_steps
        od = torch.empty((DECODE.n_seq, DECODE.H, DECODE.d), dtype=torch.bfloat16, device=dev)
        ins = [[dd[n][s] for n in ("q", "k", "v", "z", "beta")] for s in range(nsteps)]
        for s in range(3):
            kda.recurrent_step(*ins[s], dd["dt_bias"], dd["A_log"], st, out=od)
        torch.cuda.synchronize()
        dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nsteps)]
        for e_a, e_b in dev_ev:
            e_a.record(stream)
            e_b.record(stream)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk2:
            for s in range(nsteps):
                kda.set_profile_events(list(dev_ev[s]))
                kda.recurrent_step(*ins[s], dd["dt_bias"], dd["A_log"], st, out=od)
            kda.set_profile_events([])
            torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        dts = [a_.elapsed_time(b_) for a_, b_ in dev_ev]
        dms = sum(dts) / len(dts)
        dbytes = decode_bytes(DECODE.n_seq, DECODE.H, DECODE.d, 2)
        gbs = dbytes / (dms / 1e3) / 1e9
        dec = {"workload": DECODE.name, "steps": nsteps, "us_per_step": dms * 1e3,
               "GB_per_s": gbs, "bytes_per_step": dbytes,
               "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                            "traffic": None, "kernel": "decode_step"},
               "clocks": clk2.summary()}
        del dd, ins, st

        # ---------------- speculative decoding with replay (section 5.4): one call per window, the
        # state crossing HBM once where single steps would move it once per token
        Rw, Mw = 3, 4  # accepted cached drafts replayed; bonus token + 3 new drafts (bonus committed)
        dd2 = syn.make_decode(DECODE, seed=40 + rank, device=dev, steps=Rw + Mw)
        win = lambda name, a_, b_: dd2[name][a_:b_].transpose(0, 1).contiguous()  # noqa: E731
        cached = tuple(win(n_, 0, Rw) for n_ in ("q", "k", "z", "v", "beta"))
        new = tuple(win(n_, Rw, Rw + Mw) for n_ in ("q", "k", "z", "v", "beta"))
        nr_t = torch.full((DECODE.n_seq,), Rw, dtype=torch.int32, device=dev)
        nc_t = torch.ones((DECODE.n_seq,), dtype=torch.int32, device=dev)
        orp = torch.empty((DECODE.n_seq, Mw, DECODE.H, DECODE.d), dtype=torch.bfloat16, device=dev)

        def call():
            kda.recurrent_replay(cached, nr_t, new, nc_t, dd2["dt_bias"], dd2["A_log"], dd2["state"], out=orp)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        ra, rb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rts = []
        for _ in range(args.steps):  # the 512 MiB of states exceed L2
            ra.record(stream)
            call()
            rb.record(stream)
            rb.synchronize()
            rts.append(ra.elapsed_time(rb))
        rms = sum(rts) / len(rts)
        nh = DECODE.n_seq * DECODE.H
        rbytes = (2 * nh * DECODE.d * DECODE.d * 4 + (Rw + Mw) * nh * (4 * DECODE.d * 2 + 2)
                  + Mw * nh * DECODE.d * 2)
        rgb = rbytes / (rms / 1e3) / 1e9
        dec["replay"] = {"window": {"replayed": Rw, "new": Mw, "committed_new": 1},
                         "us_per_call": rms * 1e3, "tokens_per_call": DECODE.n_seq * (Rw + Mw),
                         "bytes_per_call": rbytes, "GB_per_s": rgb,
                         "roofline": {"bound": "hbm", "achieved": rgb, "peak": hbm, "unit": "GB/s",
                                      "frac": rgb / hbm, "kernel": "replay",
                                      "traffic": measured_traffic("replay", p_items=nh)},
                         "single_steps_us": (Rw + Mw) * dms * 1e3,
                         "speedup_vs_single_steps": (Rw + Mw) * dms / rms}
        del dd2, cached, new

    # ---------------- the backward pass on the headline batch (one-pass workspace, ~0.42 MiB per chunk-head);
    # last, so that its 32 GB scratch does not shape the placement of the buffers timed above
    bwd_batch = None
    if not args.no_backward:
        db = syn.make_prefill_shard(WORKLOAD, 2, rank, ws, device=dev)
        Tb, Nb = sum(db["lengths"]), len(db["lengths"])
        qb, kb, vb, zb, betab = (db[n] for n in ("q", "k", "v", "z", "beta"))
        gen = torch.Generator(device=dev).manual_seed(79 + rank)
        go_h = torch.randn(vb.shape, generator=gen, device=dev).to(vb.dtype)
        gST_h = torch.randn((Nb, H, D, D), generator=gen, device=dev) * 0.1
        need_h = kda.chunk_bwd_workspace_size(Tb, Nb, H, D, D)
        work_h = torch.empty((need_h,), dtype=torch.uint8, device=dev)

        def step_bh():
            return kda.chunk_bwd(qb, kb, vb, zb, betab, db["dt_bias"], db["A_log"], go_h, g_min=db["g_min"],
                                 scale=db["scale"], cu_seqlens=db["cu_seqlens"], initial_state=db["initial_state"],
                                 grad_final_state=gST_h, workspace=work_h)

        for _ in range(2):
            g_ = step_bh()
            del g_
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        ha, hb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hts = []
        for _ in range(3):
            ha.record(stream)
            g_ = step_bh()
            hb.record(stream)
            hb.synchronize()
            hts.append(ha.elapsed_time(hb))
            del g_
        msbh = max_over_ranks(sum(hts) / len(hts), ws)
        bwd_batch = {"what": "kda_chunk_bwd on the headline batch: d q, k, v, z, beta, dt_bias, A_log, S0 "
                             "from d o and d S_T (inputs larger than L2)",
                     "ms_per_step": msbh, "tokens_per_s": Tb / (msbh / 1e3), "vs_forward": msbh / ms_head,
                     "workspace_bytes": int(need_h)}
        del go_h, gST_h, work_h, qb, kb, vb, zb, betab, db
        torch.cuda.empty_cache()

    # ---------------- CPU oracle baseline (rank 0, N = 1 only): a seeded sample of the headline workload
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        dc = syn.make_prefill_shard(WORKLOAD, 2, 0, 1, device="cpu")
        units, th = oracle_sample_units(dc["lengths"], H)
        secs, used, total, reps = cpu_oracle_run(dc, units=units)
        cpu = {"value": th / H / secs, "unit": "tokens/s", "cores": used, "kind": "oracle",
               "sample": f"{len(units)} seeded (sequence, head) units of the varlen batch ({th} token-heads), "
                         f"best of {reps} runs, {total:.1f} s total; value = token-heads/s / {H} heads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(WORKLOAD, lengths, ws),
            "schedule": schedule_name(sch),
            "tflops": tflops, "tflops_dense_tile": fl["dense_tile"] / (ms_head / 1e3) / 1e12,
            "frac_bf16_peak": tflops / tc, "hbm_gbs_algorithmic": by["total"] / (ms_head / 1e3) / 1e9,
            "frac_hbm_algorithmic": by["total"] / (ms_head / 1e3) / 1e9 / hbm,
            "kernels_ms": dict(zip(names, kern_avg)),
            "ms_per_step_with_kernel_marks": sum(step_ms_marked) / len(step_ms_marked),
            "step_ms_min_median_max": step_spread,
            "roofline": roof,
            "e2e": {"value": T_all / (e2e_pipe_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_pipe_ms, "wall_ms_per_step": e2e_pipe_wall_ms,
                    "how": "double-buffered: step s+1's inputs (q, k, v, z, beta, initial states) copied from "
                           "pinned host memory while step s computes, step s's o and final states read back "
                           "meanwhile; every step's inputs and results cross the host link",
                    "serial": {"value": T_all / (e2e_ms / 1e3), "ms_per_step": e2e_ms,
                               "how": "copy in, compute, copy out, one step at a time, L2 flushed"}},
            "gpu_launches": nk * args.steps,
            "clocks": clocks,
            "latency_4k": lat,
            "decode": dec,
            "epilogue": epi,
            "gate_variant": gvar,
            "backward": bwd,
            "backward_batch": bwd_batch,
            "long_workloads": longw,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_case(args):
    """Small fixed cases for profiler captures (a few untimed launches, then a one-line summary).

    prefill_small: B=1, H=8, T=16384, bf16, d=128 (inputs 33.6 MB, packets 155 MB: above L2).
    prefill_4k:    the benchmark's prefill workload, B=1, H=32, T=4096, bf16, d=128.
    decode_small:  N=64 sequences x H=32 heads, d=128, fp32 state 268 MB (above L2), 8 steps.
    replay_256:    the decode workload's 256 x 32 states, one replay window (3 replayed, 4 new), 3 calls.
    softplus_4k:   the T=4096 prefill workload with the softplus gate (fp32 path), 2 calls.
    backward_4k:   the backward pass on the T=4096 prefill workload, 2 calls.
    """
    from linear_attention_kda_gb300 import build as kbuild, kda
    kbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.case == "replay_256":
        w = syn.DECODE_256
        Rw, Mw = 3, 4
        dd = syn.make_decode(w, seed=40, device=dev, steps=Rw + Mw)
        win = lambda name, a_, b_: dd[name][a_:b_].transpose(0, 1).contiguous()  # noqa: E731
        cached = tuple(win(n_, 0, Rw) for n_ in ("q", "k", "z", "v", "beta"))
        new = tuple(win(n_, Rw, Rw + Mw) for n_ in ("q", "k", "z", "v", "beta"))
        nr = torch.full((w.n_seq,), Rw, dtype=torch.int32, device=dev)
        nc = torch.ones((w.n_seq,), dtype=torch.int32, device=dev)
        for _ in range(3):
            kda.recurrent_replay(cached, nr, new, nc, dd["dt_bias"], dd["A_log"], dd["state"])
    elif args.case in ("softplus_4k", "backward_4k"):
        w = syn.PREFILL_4K
        d = syn.make_prefill(w, seed=1, device=dev)
        args_ = [d[n] for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log")]
        for _ in range(2):
            if args.case == "softplus_4k":
                kda.chunk_fwd(*args_, cu_seqlens=d["cu_seqlens"], output_final_state=True, gate="softplus")
            else:
                kda.chunk_bwd(*args_, torch.ones_like(d["v"]), cu_seqlens=d["cu_seqlens"])
    elif args.case == "intra_sep":
        # 200 sequences x 256 tokens, H = 16 (more sequences than the one-launch schedules take: the
        # intra-chunk kernel runs alone); inputs 0.84 GB, packets 0.96 GB
        w = syn.Workload("intra_sep_bf16_N200_T256_H16_d128", H=16, d=128, dtype="bf16", n_seq=200, seq_len=256,
                         z_std=1.5, b_range=1.0, alog_std=0.25)
        d = syn.make_prefill(w, seed=1, device=dev)
        for _ in range(2):
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["dt_bias"], d["A_log"],
                          cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens"].cpu(), output_final_state=True)
    elif args.case == "output_gate":
        # the Eq. 6 epilogue pass alone on 131072 tokens x 32 heads (o, g, y: 1.07 GB each)
        w = syn.Workload("output_gate_bf16_T131072_H32_d128", H=32, d=128, dtype="bf16", seq_len=131072)
        o_ = torch.randn(131072, 32, 128, device=dev).to(torch.bfloat16)
        g_, w_ = syn.make_output_gate_inputs(131072, 32, 128, "bf16", 5, device=dev)
        y_ = torch.empty_like(o_)
        for _ in range(3):
            kda.output_gate(o_, g_, w_, 1e-6, out=y_)
    elif args.case in ("prefill_small", "prefill_4k"):
        if args.case == "prefill_small":
            w = syn.Workload("prefill_small_bf16_T16384_H8_d128", H=8, d=128, dtype="bf16", seq_len=16384,
                             z_std=1.5, b_range=1.0, alog_std=0.25)
        else:
            w = syn.PREFILL_4K
        d = syn.make_prefill(w, seed=1, device=dev)
        for _ in range(3):
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["dt_bias"], d["A_log"],
                          cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens"].cpu(),
                          output_final_state=True)
    else:
        w = syn.Workload("decode_small_bf16_N64_H32_d128", H=32, d=128, dtype="bf16", n_seq=64, seq_len=1,
                         z_std=1.5, b_range=1.0, alog_std=0.25, s0_std=0.02, decode_steps=8)
        d = syn.make_decode(w, seed=4, device=dev)
        for s_ in range(8):
            kda.recurrent_step(d["q"][s_], d["k"][s_], d["v"][s_], d["z"][s_], d["beta"][s_], d["dt_bias"],
                               d["A_log"], d["state"])
    torch.cuda.synchronize()
    print(json.dumps({"case": args.case, "workload": w.name, "device_error": kda.get_device_error()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-epilogue", action="store_true")
    ap.add_argument("--no-gate-variant", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-long", action="store_true")
    ap.add_argument("--case", choices=["prefill_small", "prefill_4k", "decode_small", "replay_256", "softplus_4k",
                                       "backward_4k", "intra_sep", "output_gate"], default=None,
                    help="run a small fixed case for profiler captures instead of the benchmark")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, ws)
    else:
        run_ours(args, rank, ws, local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
