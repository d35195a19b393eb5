"""GPU parity of the unbounded softplus gate (KDA_GATE_SOFTPLUS) against the fp64 oracle.

The gate is g = -exp(A_log) * Softplus(z + b), the earlier design that the Kimi K3 report
(section 2.1.1) replaces by the bounded Eq. 5.  With it the prefill runs on the fp32 CUDA-core
path, whose in-chunk decays are exp(G_r - G_i) <= 1, so any gate magnitude is safe; decode and
replay compute the gate in their token loops.  The oracle is the fp64 token recurrence with
``gate_softplus`` (exact for any gate).  Tolerances as everywhere: 1e-2 for bf16 I/O, 1e-4 fp32.
"""
import numpy as np
import pytest
import torch

from linear_attention_kda_gb300 import kda, synthetic as syn
from oracle import numpy_ref as R
from tests.gpu_util import TOL_BF16, TOL_F32, compare_prefill, rel_err, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev(cuda_ok):
    torch.cuda.set_device(0)
    kda.load_library()


def _varlen(H, D, dtype, lengths, seed, z_std=1.5, alog_std=0.25, alog_mean=0.0, s0_std=0.02):
    T = sum(lengths)
    q, k, v, beta, z = syn.make_tokens(T, H, D, D, dtype, seed, z_std=z_std)
    b, a = syn.make_head_params(H, D, seed, b_range=1.0, alog_std=alog_std)
    d = dict(q=q, k=k, v=v, beta=beta, z=z, dt_bias=b, A_log=a + alog_mean, g_min=-5.0, scale=1.0,
             lengths=lengths, cu_seqlens=syn.cu_seqlens_of(lengths))
    d["initial_state"] = syn.make_state(len(lengths), H, D, D, s0_std, seed) if s0_std > 0 else None
    return d


def _oracle(d):
    f = lambda name: d[name].double().numpy()  # noqa: E731  (inputs as the kernel reads them)
    s0 = d["initial_state"]
    o, ST = R.forward(f("q"), f("k"), f("v"), f("z"), f("beta"), f("dt_bias"), f("A_log"), d["cu_seqlens"],
                      S0=None if s0 is None else s0.double().numpy(), scale=d["scale"], gate_kind="softplus")
    cu = [int(x) for x in d["cu_seqlens"]]
    H = d["q"].shape[1]
    return {(n, h): (o[cu[n]:cu[n + 1], h], ST[n, h]) for n in range(len(cu) - 1) for h in range(H)}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_softplus_elementwise_and_chunk_cumsum(dtype):
    lengths = [5, 0, 64, 65, 130, 1]
    T, H, D = sum(lengths), 3, 128
    _, _, _, _, z = syn.make_tokens(T, H, D, D, dtype, 5, z_std=3.0)
    b, a = syn.make_head_params(H, D, 5, b_range=1.0, alog_std=0.5)
    g = kda.gate(z.cuda(), b.cuda(), a.cuda(), gate="softplus").cpu().numpy()
    ref = R.gate_softplus(z.float().numpy(), b.numpy()[None], a.numpy()[None, :, None])
    np.testing.assert_allclose(g, ref, rtol=2e-6, atol=1e-7)
    assert np.all(g < 0)
    assert g.min() < -5.0  # unbounded: below the bounded gate's floor on this draw
    cu = syn.cu_seqlens_of(lengths)
    G = kda.gate(z.cuda(), b.cuda(), a.cuda(), chunk_size=64, cu_seqlens=cu.cuda(), gate="softplus").cpu().numpy()
    assert kda.get_device_error() == 0
    Gref = np.zeros_like(ref)
    for n in range(len(lengths)):
        for c0 in range(int(cu[n]), int(cu[n + 1]), 64):
            c1 = min(c0 + 64, int(cu[n + 1]))
            Gref[c0:c1] = np.cumsum(ref[c0:c1], axis=0)
    np.testing.assert_allclose(G, Gref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f32"), (128, "f32")])
def test_prefill_softplus_matches_oracle(D, dtype):
    """Ragged varlen batch (empty, 1, 63, 64, 65, 130, 200 tokens) with initial and final states."""
    d = _varlen(3, D, dtype, [1, 63, 64, 65, 200, 0, 130], seed=31)
    cu = d["cu_seqlens"]
    sch = kda.chunk_fwd_schedule(int(cu[-1]), len(cu) - 1, 3, D, D,
                                 torch.bfloat16 if dtype == "bf16" else torch.float32, cu, gate="softplus")
    assert not sch["fused"] and sch["seg_len"] == 0 and sch["kernels"] == 3  # the fp32 CUDA-core path
    o, fs = run_prefill(d, gate="softplus")
    compare_prefill(d, o, fs, _oracle(d), TOL_F32 if dtype == "f32" else TOL_BF16)


def test_prefill_softplus_extreme_decays():
    """exp(A) ~ 55 and wide logits: per-token log-decays reach the hundreds, so states are wiped
    within a token (alpha underflows to 0).  A factored Gamma / (1/Gamma) form would overflow here;
    the result must stay finite and match the oracle."""
    d = _varlen(2, 128, "bf16", [200, 77], seed=32, z_std=3.0, alog_mean=4.0)
    g = R.gate_softplus(d["z"].float().numpy(), d["dt_bias"].numpy()[None], d["A_log"].numpy()[None, :, None])
    assert g.min() < -300.0 and np.mean(g < -88.0) > 0.2  # many decays below fp32's exp range
    o, fs = run_prefill(d, gate="softplus")
    assert torch.isfinite(o).all() and torch.isfinite(fs).all()
    compare_prefill(d, o, fs, _oracle(d), TOL_BF16)


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f32")])
def test_recurrent_step_softplus_matches_oracle(D, dtype):
    w = syn.Workload("dsp", H=3, d=D, dtype=dtype, n_seq=4, seq_len=1, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02, decode_steps=5)
    d = syn.make_decode(w, seed=33)
    N, H, S = 4, 3, 5
    st = d["state"].clone().cuda()
    outs = []
    for s in range(S):
        args = [d[n][s].contiguous().cuda() for n in ("q", "k", "v", "z", "beta")]
        outs.append(kda.recurrent_step(*args, d["dt_bias"].cuda(), d["A_log"].cuda(), st, gate="softplus").float().cpu())
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for n in range(N):
        for h in range(H):
            seq = lambda name: torch.stack([d[name][s][n, h] for s in range(S)]).double().numpy()  # noqa: E731
            g = R.gate_softplus(seq("z"), d["dt_bias"][h].double().numpy(), float(d["A_log"][h]))
            o_ref, S_ref = R.recurrence(seq("q"), seq("k"), seq("v"), g, seq("beta"), S0=d["state"][n, h].double().numpy())
            assert rel_err(torch.stack([outs[s][n, h] for s in range(S)]).numpy(), o_ref) <= tol, (n, h)
            assert rel_err(st[n, h].cpu().numpy(), S_ref) <= tol, (n, h)


def test_recurrent_replay_softplus_matches_oracle():
    D, N, H, Rw, M = 128, 5, 2, 3, 4
    w = syn.Workload("rsp", H=H, d=D, dtype="bf16", n_seq=N, seq_len=1, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02, decode_steps=Rw + M)
    d = syn.make_decode(w, seed=34)
    win = lambda name, a, b: d[name][a:b].transpose(0, 1).contiguous()  # noqa: E731
    cached = tuple(win(n, 0, Rw) for n in ("q", "k", "z", "v", "beta"))
    new = tuple(win(n, Rw, Rw + M) for n in ("q", "k", "z", "v", "beta"))
    nr = torch.tensor([3, 0, 2, 1, 3], dtype=torch.int32)
    nc = torch.tensor([1, 2, 0, 4, 1], dtype=torch.int32)
    st = d["state"].clone().cuda()
    o = kda.recurrent_replay(tuple(x.cuda() for x in cached), nr.cuda(), tuple(x.cuda() for x in new), nc.cuda(),
                             d["dt_bias"].cuda(), d["A_log"].cuda(), st, gate="softplus").float().cpu()
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0

    def tup(t, n, h):
        q, k, z, v, beta = (x[n, :, h].double().numpy() for x in t)
        return q, k, v, R.gate_softplus(z, d["dt_bias"][h].double().numpy(), float(d["A_log"][h])), beta

    for n in range(N):
        for h in range(H):
            o_ref, S_ref = R.replay(tup(cached, n, h), int(nr[n]), tup(new, n, h), int(nc[n]),
                                    d["state"][n, h].double().numpy())
            assert rel_err(o[n, :, h].numpy(), o_ref) <= TOL_BF16, (n, h)
            assert rel_err(st[n, h].cpu().numpy(), S_ref) <= TOL_BF16, (n, h)


def test_bounded_gate_below_tensor_core_range_runs_fp32_path():
    """Eq. 5 with g_min = -8 and bf16 d = 128: the tensor-core prefill scales rows and keys by
    e^{G_r - G_p} against references up to 16 tokens away, which leaves fp32 range once 16 |g_min|
    exceeds ~88, so kda_chunk_fwd takes the fp32 path (3 kernels, the fp32 path's workspace).  The
    logits are shifted so that most decays sit near the bound; results against the fp64 oracle."""
    from tests.gpu_util import oracle_prefill
    d = _varlen(2, 128, "bf16", [200, 77, 64], seed=63)
    d["z"] = (d["z"].float() + 4.0).to(d["z"].dtype)
    d["g_min"] = -8.0
    assert kda.chunk_fwd_kernel_count(sum(d["lengths"]), 3, 2, 128, 128, torch.bfloat16, d["cu_seqlens"],
                                      g_min=-8.0) == 3
    assert kda.chunk_fwd_workspace_size(sum(d["lengths"]), 3, 2, 128, 128, torch.bfloat16, 64, d["cu_seqlens"],
                                        g_min=-8.0) == \
        kda.chunk_fwd_workspace_size(sum(d["lengths"]), 3, 2, 128, 128, torch.bfloat16, 64, d["cu_seqlens"],
                                     gate="softplus")
    o, fs = run_prefill(d)
    assert torch.isfinite(o).all() and torch.isfinite(fs).all()
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16)
