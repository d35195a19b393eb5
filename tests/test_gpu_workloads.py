"""Parity at the full sizes of the benchmark workloads, on sampled outputs.

The GPU path runs each workload at full size (same launch path as the
benchmark); the fp64 oracle recomputes a seeded sample of (sequence, head)
units one by one.  Tolerance: relative Frobenius error <= 1e-2 per unit on
outputs and final states (bf16 I/O, fp32 accumulation).
"""
import random

import numpy as np
import pytest
import torch

from linear_attention_kda_gb300 import kda, synthetic as syn
from oracle import c_ref
from tests.gpu_util import TOL_BF16, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev(cuda_ok):
    torch.cuda.set_device(0)
    kda.load_library()


def _run(d, dev="cuda"):
    o, fs = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["dt_bias"].to(dev), d["A_log"].to(dev),
                          g_min=d["g_min"], scale=d["scale"], cu_seqlens=d["cu_seqlens"].to(dev),
                          cu_seqlens_host=d["cu_seqlens"].cpu(),
                          initial_state=None if d["initial_state"] is None else d["initial_state"].to(dev),
                          output_final_state=True)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return o, fs


def _unit_inputs(d, n, h):
    """fp32 CPU copies of one (sequence, head) unit's inputs."""
    cu = [int(x) for x in d["cu_seqlens"].cpu()]
    a, b = cu[n], cu[n + 1]
    sl = lambda x: x[a:b, h:h + 1].float().cpu().contiguous()  # noqa: E731
    return dict(q=sl(d["q"]), k=sl(d["k"]), v=sl(d["v"]), z=sl(d["z"]),
                beta=d["beta"][a:b, h:h + 1].float().cpu().contiguous(),
                b=d["dt_bias"][h:h + 1].cpu(), A=d["A_log"][h:h + 1].cpu(),
                s0=None if d["initial_state"] is None else d["initial_state"][n:n + 1, h:h + 1].cpu(),
                span=(a, b))


def _oracle_units(d, units, nthreads=None):
    """Runs the C oracle on each unit separately (inputs sliced to one head)."""
    out = {}
    probs = []
    for n, h in units:
        u = _unit_inputs(d, n, h)
        L = u["span"][1] - u["span"][0]
        probs.append((n, h, u, L))
    # one call per unit keeps host memory bounded; the C oracle is parallel across units of a call
    for n, h, u, L in probs:
        res, _ = c_ref.forward(u["q"], u["k"], u["v"], u["z"], u["beta"], u["b"], u["A"], [0, L],
                               S0=u["s0"], g_min=d["g_min"], scale=d["scale"], nthreads=nthreads)
        out[(n, h)] = res[(0, 0)]
    return out


def test_varlen_workload_sampled_units():
    """32 sequences, lengths U[512, 8192] (~140K tokens), H=32, random initial states."""
    d = syn.make_prefill(syn.VARLEN_32, seed=2, device="cuda")
    assert len(d["lengths"]) == 32 and 512 <= min(d["lengths"]) and max(d["lengths"]) <= 8192
    o, fs = _run(d)
    assert torch.isfinite(o.float()).all() and torch.isfinite(fs).all()
    rng = random.Random(2)
    units = sorted({(rng.randrange(32), rng.randrange(32)) for _ in range(24)})
    # always include the shortest and the longest sequence
    lens = d["lengths"]
    units += [(int(np.argmin(lens)), 0), (int(np.argmax(lens)), 31)]
    ref = _oracle_units(d, units)
    cu = [int(x) for x in d["cu_seqlens"].cpu()]
    for (n, h), (o_ref, S_ref) in ref.items():
        eo = rel_err(o[cu[n]:cu[n + 1], h].float().cpu().numpy(), o_ref)
        es = rel_err(fs[n, h].cpu().numpy(), S_ref)
        assert eo <= TOL_BF16 and es <= TOL_BF16, (n, h, eo, es)


def test_long_context_workload_sampled_heads():
    """B=1, H=32, T=1,048,576: 2 sampled heads checked in full, plus every head's final state
    after the first 16K tokens (a separate 16K-token call on the same inputs)."""
    w = syn.LONG_1M
    d = syn.make_prefill(w, seed=3, device="cuda")
    o, fs = _run(d)
    assert torch.isfinite(fs).all()
    rng = random.Random(3)
    heads = rng.sample(range(w.H), 2)
    # both sampled heads in one oracle call (one host thread each)
    hs = torch.tensor(heads, device="cuda")
    pick = lambda x: x.index_select(1, hs).float().cpu().contiguous()  # noqa: E731
    res, _ = c_ref.forward(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["z"]), pick(d["beta"]),
                           d["dt_bias"][heads].cpu(), d["A_log"][heads].cpu(), [0, w.seq_len],
                           g_min=d["g_min"], scale=d["scale"])
    for i, h in enumerate(heads):
        o_ref, S_ref = res[(0, i)]
        eo = rel_err(o[:, h].float().cpu().numpy(), o_ref)
        es = rel_err(fs[0, h].cpu().numpy(), S_ref)
        assert eo <= TOL_BF16 and es <= TOL_BF16, (h, eo, es)
    del o, fs
    # first 16K tokens, all heads: final states
    T16 = 1 << 14
    d16 = dict(d)
    for nm in ("q", "k", "v", "z", "beta"):
        d16[nm] = d[nm][:T16].contiguous()
    d16["cu_seqlens"] = torch.tensor([0, T16], dtype=torch.int32)
    o16, fs16 = _run(d16)
    del d
    torch.cuda.empty_cache()
    res, _ = c_ref.forward(d16["q"], d16["k"], d16["v"], d16["z"], d16["beta"], d16["dt_bias"], d16["A_log"],
                           [0, T16], g_min=d16["g_min"], scale=d16["scale"])
    for h in range(w.H):
        o_ref, S_ref = res[(0, h)]
        assert rel_err(fs16[0, h].cpu().numpy(), S_ref) <= TOL_BF16, h
        assert rel_err(o16[:, h].float().cpu().numpy(), o_ref) <= TOL_BF16, h


def test_decode_workload_equals_prefill():
    """256 sequences x 32 heads, 512 in-place decode steps == kda_chunk_fwd over the same 512 tokens
    from the same states; a seeded subset of units is also checked against the oracle."""
    w = syn.DECODE_256
    d = syn.make_decode(w, seed=4, device="cuda")
    N, H, S = w.n_seq, w.H, w.decode_steps
    S0 = d["state"].clone()
    st = d["state"]
    o_dec = torch.empty((S, N, H, w.d), dtype=torch.bfloat16, device="cuda")
    for s in range(S):
        kda.recurrent_step(d["q"][s], d["k"][s], d["v"][s], d["z"][s], d["beta"][s], d["dt_bias"], d["A_log"], st,
                           out=o_dec[s])
    torch.cuda.synchronize()
    err = kda.get_device_error()
    assert err == 0, f"device error {err} after the decode steps"
    seq = lambda x: x.transpose(0, 1).reshape(N * S, *x.shape[2:]).contiguous()  # noqa: E731
    cu = torch.arange(0, N * S + 1, S, dtype=torch.int32)
    o_pf, fs_pf = kda.chunk_fwd(seq(d["q"]), seq(d["k"]), seq(d["v"]), seq(d["z"]), seq(d["beta"]),
                                d["dt_bias"], d["A_log"], cu_seqlens=cu.cuda(), cu_seqlens_host=cu,
                                initial_state=S0, output_final_state=True)
    torch.cuda.synchronize()
    err = kda.get_device_error()
    assert err == 0, f"device error {err} after the prefill"
    o_pf = o_pf.view(N, S, H, w.d)
    o_dec_n = o_dec.transpose(0, 1)
    # every (sequence, head): decode vs prefill
    num_o = (o_dec_n.float() - o_pf.float()).pow(2).sum(dim=(1, 3)).sqrt()
    den_o = o_pf.float().pow(2).sum(dim=(1, 3)).sqrt()
    eo = num_o / den_o
    assert float(eo.max()) <= TOL_BF16, f"o: max rel err {float(eo.max()):.3g} at {divmod(int(eo.argmax()), H)}"
    num_s = (st - fs_pf).pow(2).sum(dim=(2, 3)).sqrt()
    den_s = fs_pf.pow(2).sum(dim=(2, 3)).sqrt()
    es = num_s / den_s
    assert float(es.max()) <= TOL_BF16, f"S: max rel err {float(es.max()):.3g} at {divmod(int(es.argmax()), H)}"
    # seeded subset against the oracle
    rng = random.Random(4)
    units = sorted({(rng.randrange(N), rng.randrange(H)) for _ in range(12)})
    dd = dict(q=seq(d["q"]), k=seq(d["k"]), v=seq(d["v"]), z=seq(d["z"]), beta=seq(d["beta"]),
              dt_bias=d["dt_bias"].cpu(), A_log=d["A_log"].cpu(), initial_state=S0.cpu(), cu_seqlens=cu,
              g_min=d["g_min"], scale=d["scale"])
    ref = _oracle_units(dd, units)
    for (n, h), (o_ref, S_ref) in ref.items():
        assert rel_err(o_dec_n[n, :, h].float().cpu().numpy(), o_ref) <= TOL_BF16
        assert rel_err(st[n, h].cpu().numpy(), S_ref) <= TOL_BF16
