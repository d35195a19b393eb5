"""Helpers for the GPU parity tests: run libkda on seeded inputs, compare with the oracle."""
import numpy as np
import torch

from linear_attention_kda_gb300 import kda
from oracle import c_ref

TOL_BF16 = 1e-2  # relative Frobenius error per head, bf16 I/O, fp32 accumulation
TOL_F32 = 1e-4   # relative Frobenius error per head, fp32 path


def rel_err(x, ref) -> float:
    """||x - ref||_F / ||ref||_F (absolute error when ||ref||_F < 1e-30)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    d = float(np.linalg.norm(x - ref))
    n = float(np.linalg.norm(ref))
    return d / n if n >= 1e-30 else d


def run_prefill(d, dev="cuda", *, with_state=True, heads=None, **kw):
    """Runs kda_chunk_fwd on a synthetic input dict (CPU tensors). Returns (o, final_state) on CPU."""
    sel = (lambda x: x) if heads is None else (lambda x: x[:, heads].contiguous())
    q, k, v, z, beta = (sel(d[n]).to(dev) for n in ("q", "k", "v", "z", "beta"))
    b = d["dt_bias"] if heads is None else d["dt_bias"][heads].contiguous()
    a = d["A_log"] if heads is None else d["A_log"][heads].contiguous()
    s0 = d.get("initial_state")
    if s0 is not None and heads is not None:
        s0 = s0[:, heads].contiguous()
    o, fs = kda.chunk_fwd(q, k, v, z, beta, b.to(dev), a.to(dev), g_min=d["g_min"], scale=d["scale"],
                          cu_seqlens=d["cu_seqlens"].to(dev), cu_seqlens_host=d["cu_seqlens"],
                          initial_state=None if s0 is None else s0.to(dev),
                          output_final_state=with_state, **kw)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return o.float().cpu(), (fs.cpu() if fs is not None else None)


def oracle_prefill(d, units=None, heads=None):
    sel = (lambda x: x) if heads is None else (lambda x: x[:, heads].contiguous())
    b = d["dt_bias"] if heads is None else d["dt_bias"][heads]
    a = d["A_log"] if heads is None else d["A_log"][heads]
    s0 = d.get("initial_state")
    if s0 is not None and heads is not None:
        s0 = s0[:, heads]
    res, _ = c_ref.forward(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["z"]), sel(d["beta"]), b, a,
                           d["cu_seqlens"], S0=s0, g_min=d["g_min"], scale=d["scale"], units=units)
    return res


def compare_prefill(d, o, fs, res, tol):
    """Max per-(sequence, head) relative error of o and final state vs oracle results."""
    cu = [int(x) for x in d["cu_seqlens"]]
    worst = 0.0
    for (n, h), (o_ref, S_ref) in res.items():
        a, b = cu[n], cu[n + 1]
        eo = rel_err(o[a:b, h].numpy(), o_ref) if b > a else 0.0
        es = rel_err(fs[n, h].numpy(), S_ref) if fs is not None else 0.0
        assert np.isfinite(eo) and np.isfinite(es)
        assert eo <= tol and es <= tol, f"(seq {n}, head {h}): rel err o={eo:.3g} S={es:.3g} tol={tol}"
        worst = max(worst, eo, es)
    return worst
