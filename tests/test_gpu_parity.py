"""GPU parity of libkda against the fp64 oracle (through the C ABI).

Tolerances (relative Frobenius error per (sequence, head), on outputs and
final states): 1e-2 for bf16 I/O with fp32 accumulation, 1e-4 for the fp32
path.  Inputs are the seeded synthetic workloads (same distributions as the
benchmark), shortened where the oracle must run on every head.
"""
import numpy as np
import pytest
import torch

from linear_attention_kda_gb300 import kda, synthetic as syn
from oracle import c_ref, numpy_ref as R
from tests.gpu_util import TOL_BF16, TOL_F32, compare_prefill, oracle_prefill, rel_err, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev(cuda_ok):
    torch.cuda.set_device(0)
    kda.load_library()


def _varlen(w, lengths, seed, s0_std=None):
    d = syn.make_prefill(w, seed, T_override=1)
    T = sum(lengths)
    q, k, v, beta, z = syn.make_tokens(T, w.H, w.d, w.d, w.dtype, seed, z_std=w.z_std)
    d.update(q=q, k=k, v=v, beta=beta, z=z, lengths=lengths, cu_seqlens=syn.cu_seqlens_of(lengths))
    std = w.s0_std if s0_std is None else s0_std
    d["initial_state"] = syn.make_state(len(lengths), w.H, w.d, w.d, std, seed) if std > 0 else None
    return d


# ----------------------------------------------------------------------------- gate

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_elementwise(dtype):
    w = syn.PREFILL_4K
    d = syn.make_prefill(syn.Workload("g", H=3, d=128, dtype=dtype, seq_len=100, z_std=3.0,
                                      b_range=1.0, alog_std=0.5), seed=3)
    g = kda.gate(d["z"].cuda(), d["dt_bias"].cuda(), d["A_log"].cuda(), g_min=-5.0).cpu().numpy()
    ref = R.gate(d["z"].float().numpy(), d["dt_bias"].numpy()[None], d["A_log"].numpy()[None, :, None])
    np.testing.assert_allclose(g, ref, rtol=1e-5, atol=1e-6)
    assert np.all(g >= -5.0) and np.all(g <= 0.0)
    assert w.H == 32


def test_gate_chunk_cumsum_varlen():
    lengths = [5, 0, 64, 65, 130, 1, 200]
    w = syn.Workload("g", H=2, d=64, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0, alog_std=0.25)
    T = sum(lengths)
    q, k, v, beta, z = syn.make_tokens(T, 2, 64, 64, "bf16", 9, z_std=1.5)
    b, a = syn.make_head_params(2, 64, 9, b_range=1.0, alog_std=0.25)
    cu = syn.cu_seqlens_of(lengths)
    G = kda.gate(z.cuda(), b.cuda(), a.cuda(), chunk_size=64, cu_seqlens=cu.cuda()).cpu().numpy()
    assert kda.get_device_error() == 0
    g = R.gate(z.float().numpy(), b.numpy()[None], a.numpy()[None, :, None])
    ref = np.zeros_like(g)
    for n in range(len(lengths)):
        for c0 in range(int(cu[n]), int(cu[n + 1]), 64):
            c1 = min(c0 + 64, int(cu[n + 1]))
            ref[c0:c1] = np.cumsum(g[c0:c1], axis=0)
    np.testing.assert_allclose(G, ref, rtol=1e-5, atol=2e-4)
    assert w.d == 64


def test_gate_bad_seqlens_sets_device_error():
    z = torch.zeros((10, 1, 16), dtype=torch.float32, device="cuda")
    cu = torch.tensor([0, 7, 3, 10], dtype=torch.int32, device="cuda")  # not monotone
    kda.gate(z, chunk_size=4, cu_seqlens=cu)
    assert kda.get_device_error() == 7
    assert kda.get_device_error() == 0  # cleared


# ----------------------------------------------------------------------------- decode

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_recurrent_step_matches_oracle(D, dtype):
    w = syn.Workload("dec", H=3, d=D, dtype=dtype, n_seq=5, seq_len=1, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02, decode_steps=6)
    d = syn.make_decode(w, seed=11)
    N, H, S = 5, 3, 6
    # slots permuted, plus one spare slot that must stay untouched
    slots = torch.tensor([3, 0, 5, 1, 2], dtype=torch.int32)
    pool = torch.randn((6, H, D, D)) * 0.02
    pool[slots.long()] = d["state"]
    pool_gpu = pool.cuda()
    outs = []
    for s in range(S):
        args = [d[n][s].contiguous().cuda() for n in ("q", "k", "v", "z", "beta")]
        outs.append(kda.recurrent_step(*args, d["dt_bias"].cuda(), d["A_log"].cuda(), pool_gpu,
                                       state_indices=slots.cuda()).float().cpu())
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    seq = lambda n: torch.stack([d[n][s] for s in range(S)], 1).reshape(N * S, H, *d[n].shape[3:])  # noqa: E731
    cu = torch.arange(0, N * S + 1, S, dtype=torch.int32)
    res, _ = c_ref.forward(seq("q"), seq("k"), seq("v"), seq("z"), seq("beta"), d["dt_bias"], d["A_log"],
                           cu, S0=d["state"])
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    pool_out = pool_gpu.cpu()
    for n in range(N):
        for h in range(H):
            o_ref, S_ref = res[(n, h)]
            o_gpu = torch.stack([outs[s][n, h] for s in range(S)]).numpy()
            assert rel_err(o_gpu, o_ref) <= tol
            assert rel_err(pool_out[int(slots[n]), h].numpy(), S_ref) <= tol
    assert torch.equal(pool_out[4], pool[4])  # unused slot untouched


def test_recurrent_step_bad_index_reports_and_skips():
    D, H = 64, 1
    st = torch.zeros((2, H, D, D), device="cuda")
    x = torch.zeros((1, H, D), device="cuda")
    b = torch.zeros((1, H), device="cuda")
    kda.recurrent_step(x, x, x, x, b, None, None, st, state_indices=torch.tensor([5], dtype=torch.int32, device="cuda"))
    assert kda.get_device_error() == 8
    assert torch.count_nonzero(st) == 0


# ----------------------------------------------------------------------------- prefill

def test_tiny_f32_workload():
    """B=1, H=2, T=256, d=64, fp32, zero initial state: <= 1e-4 against the fp64 recurrence."""
    d = syn.make_prefill(syn.TINY_F32, seed=0)
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_F32)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 128), ("bf16", 64), ("f32", 64)])
def test_varlen_ragged_with_state(dtype, D):
    """Ragged lengths (empty, 1, chunk +-1, multi-chunk tails) with a random initial state."""
    w = syn.Workload("v", H=3, d=D, dtype=dtype, seq_len=None, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = _varlen(w, [1, 63, 64, 0, 65, 130, 200, 7], seed=21)
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_F32 if dtype == "f32" else TOL_BF16)


def test_prefill_4k_workload_full():
    """The single-sequence bf16 workload at full size (T=4096, H=32, d=128), every head."""
    d = syn.make_prefill(syn.PREFILL_4K, seed=1)
    o, fs = run_prefill(d)
    worst = compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16)
    assert worst < TOL_BF16


def test_equal_length_batch_without_cu_seqlens():
    w = syn.Workload("b", H=2, d=128, dtype="bf16", n_seq=3, seq_len=100, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = syn.make_prefill(w, seed=5)
    dev = "cuda"
    o, fs = kda.chunk_fwd(*(d[n].to(dev) for n in ("q", "k", "v", "z", "beta")), d["dt_bias"].to(dev),
                          d["A_log"].to(dev), n_seq=3, initial_state=d["initial_state"].to(dev),
                          output_final_state=True)
    compare_prefill(d, o.float().cpu(), fs.cpu(), oracle_prefill(d), TOL_BF16)


def test_final_state_aliases_initial_state():
    w = syn.Workload("a", H=2, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = _varlen(w, [70, 3, 128], seed=6)
    st = d["initial_state"].cuda().contiguous()
    dev = "cuda"
    o, fs = kda.chunk_fwd(*(d[n].to(dev) for n in ("q", "k", "v", "z", "beta")), d["dt_bias"].to(dev),
                          d["A_log"].to(dev), cu_seqlens=d["cu_seqlens"].to(dev), initial_state=st,
                          final_state=st)
    torch.cuda.synchronize()
    compare_prefill(d, o.float().cpu(), st.cpu(), oracle_prefill(d), TOL_BF16)


@pytest.mark.parametrize("dtype,D,H", [("bf16", 128, 2), ("bf16", 128, 32), ("f32", 64, 2)])
def test_empty_sequences_copy_initial_state_exactly(dtype, D, H):
    """Empty sequences among non-empty ones (Eq. 1 takes no step: S_T = S_0).  Their final state is
    their initial state bit for bit: on the fused tensor-core launch (6 x 2 chains), the separate
    tensor-core kernels (6 x 32 chains) and the fp32 path.  The other sequences match the oracle."""
    w = syn.Workload("e", H=H, d=D, dtype=dtype, seq_len=None, z_std=1.5, b_range=1.0, alog_std=0.25,
                     s0_std=0.5)
    lengths = [0, 70, 0, 0, 130, 0]
    d = _varlen(w, lengths, seed=8)
    if dtype == "bf16":
        sch = kda.chunk_fwd_schedule(sum(lengths), len(lengths), H, D, D, torch.bfloat16, d["cu_seqlens"])
        assert sch["fused"] == (H == 2)
    o, fs = run_prefill(d)
    for n, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(fs[n], d["initial_state"][n]), n
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16 if dtype == "bf16" else TOL_F32)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_empty_batch_passes_states_through(dtype, D):
    """T = 0 over three sequences (cu_seqlens all zero): the final states are the initial states bit
    for bit, or zeros without them (the buffer starts as NaN); no token pointer is read."""
    H, N = 2, 3
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    tok = lambda *s: torch.empty(s, dtype=dt, device="cuda")  # noqa: E731
    b, a = syn.make_head_params(H, D, 3, b_range=1.0, alog_std=0.25)
    S0 = syn.make_state(N, H, D, D, 0.5, 3).cuda()
    cu = torch.zeros(N + 1, dtype=torch.int32)
    args = (tok(0, H, D), tok(0, H, D), tok(0, H, D), tok(0, H, D), tok(0, H), b.cuda(), a.cuda())
    o, fs = kda.chunk_fwd(*args, cu_seqlens=cu.cuda(), cu_seqlens_host=cu, initial_state=S0,
                          output_final_state=True)
    fz = torch.full((N, H, D, D), float("nan"), device="cuda")
    kda.chunk_fwd(*args, cu_seqlens=cu.cuda(), final_state=fz)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert o.shape == (0, H, D)
    assert torch.equal(fs, S0)
    assert not torch.isnan(fz).any() and torch.count_nonzero(fz).item() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_slow_decay_correlated_keys(dtype):
    """Inputs where (I + L) is far from I: slow decays (g about -0.05 per token, so a 64-token chunk
    decays by about e^-3 only) and keys sharing a common direction (pairwise products about 0.5, so
    the spectral norm of L reaches several units).  The benchmark's gate forgets within a token or two
    and leaves L tiny; these inputs exercise the UT-transform inverse and the state pass instead.
    Two sequences (200 and 130 tokens) with an initial state, d = 128 (tensor cores for bf16)."""
    H, D, lengths = 2, 128, [200, 130]
    T = sum(lengths)
    gen = torch.Generator().manual_seed(21)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)

    base = torch.randn((1, H, D), generator=gen)
    q = unit(torch.randn((T, H, D), generator=gen)).to(dt)
    k = unit(torch.randn((T, H, D), generator=gen) + base).to(dt)
    v = torch.randn((T, H, D), generator=gen).to(dt)
    beta = torch.sigmoid(torch.randn((T, H), generator=gen)).to(dt)
    z = (torch.randn((T, H, D), generator=gen) * 0.3 - 4.6).to(dt)  # g = -5 sigmoid(z) ~ -0.05
    d = dict(q=q, k=k, v=v, beta=beta, z=z, dt_bias=torch.zeros((H, D)), A_log=torch.zeros(H),
             initial_state=torch.randn((2, H, D, D), generator=gen) * 0.02, lengths=lengths,
             cu_seqlens=syn.cu_seqlens_of(lengths), g_min=-5.0, scale=1.0)
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16 if dtype == "bf16" else TOL_F32)


@pytest.mark.parametrize("split", [1, 64, 100, 129])
def test_split_resume_matches_one_pass(split):
    """Final state of a prefix passed as the initial state of the rest equals one pass (prefix reuse)."""
    w = syn.Workload("s", H=2, d=128, dtype="bf16", seq_len=300, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = syn.make_prefill(w, seed=8)
    o_full, fs_full = run_prefill(d)
    d1 = dict(d, cu_seqlens=torch.tensor([0, split], dtype=torch.int32))
    d2 = dict(d, cu_seqlens=torch.tensor([0, 300 - split], dtype=torch.int32))
    for n in ("q", "k", "v", "z", "beta"):
        d1[n] = d[n][:split].contiguous()
        d2[n] = d[n][split:].contiguous()
    o1, fs1 = run_prefill(d1)
    d2["initial_state"] = fs1
    o2, fs2 = run_prefill(d2)
    o_cat = torch.cat([o1, o2])
    for h in range(2):
        assert rel_err(o_cat[:, h].numpy(), o_full[:, h].numpy()) <= TOL_BF16
        assert rel_err(fs2[0, h].numpy(), fs_full[0, h].numpy()) <= TOL_BF16
    compare_prefill(d, o_cat, fs2, oracle_prefill(d), TOL_BF16)


def test_zero_state_identity_gate_limits():
    """z -> -inf gives g = 0 (alpha = 1); with beta = 0 the state is carried unchanged."""
    T, H, D = 130, 2, 128
    q, k, v, beta, z = syn.make_tokens(T, H, D, D, "bf16", 12, z_std=1.0)
    z = torch.full_like(z, -1e4)
    beta = torch.zeros_like(beta)
    S0 = torch.randn((1, H, D, D)) * 0.1
    dev = "cuda"
    o, fs = kda.chunk_fwd(q.to(dev), k.to(dev), v.to(dev), z.to(dev), beta.to(dev), None, None,
                          initial_state=S0.to(dev), output_final_state=True)
    torch.cuda.synchronize()
    assert rel_err(fs.cpu().numpy(), S0.numpy()) <= 1e-6
    o_ref = torch.einsum("thc,hcj->thj", q.float(), S0[0])
    assert rel_err(o.float().cpu().numpy(), o_ref.numpy()) <= TOL_BF16


def test_fused_schedule_varlen_own_chunks():
    """Fused launch on a batch with an empty sequence where each chain first produces its own first
    chunks and the producers take the rest (their item map skips those chunks per sequence)."""
    w = syn.Workload("f", H=16, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = _varlen(w, [1000, 0, 700, 5], seed=23)
    sch = kda.chunk_fwd_schedule(sum(d["lengths"]), 4, 16, 128, 128, torch.bfloat16, d["cu_seqlens"])
    assert sch["fused"] and sch["own_chunks"] >= 1 and sch["kernels"] == 1
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16)


def test_fused_bad_cu_seqlens_reports_device_error():
    """The fused launch validates cu_seqlens itself (no planning kernel runs before it)."""
    w = syn.Workload("e", H=2, d=128, dtype="bf16", seq_len=64)
    d = syn.make_prefill(w, seed=1)
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32)
    assert kda.chunk_fwd_schedule(64, 3, 2, 128, 128, torch.bfloat16, None)["fused"]
    dev = "cuda"
    kda.chunk_fwd(*(d[n].to(dev) for n in ("q", "k", "v", "z", "beta")), None, None, cu_seqlens=cu.to(dev),
                  output_final_state=True)
    assert kda.get_device_error() == 7


def test_bad_cu_seqlens_reports_device_error():
    w = syn.Workload("e", H=1, d=64, dtype="f32", seq_len=64)
    d = syn.make_prefill(w, seed=1)
    dev = "cuda"
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device=dev)
    kda.chunk_fwd(*(d[n].to(dev) for n in ("q", "k", "v", "z", "beta")), None, None, cu_seqlens=cu,
                  output_final_state=True)
    assert kda.get_device_error() == 7


def test_decode_equals_prefill_continuation():
    """512 in-place decode steps equal kda_chunk_fwd over the same tokens from the same state
    (decode workload, reduced to 8 sequences x 4 heads x 96 steps)."""
    w = syn.DECODE_256
    N, H, S = 8, 4, 96
    d = syn.make_decode(w, seed=4, n_seq=N, steps=S)
    hs = slice(0, H)
    st = d["state"][:, hs].contiguous().cuda()
    S0 = d["state"][:, hs].contiguous()
    b, a = d["dt_bias"][hs].contiguous().cuda(), d["A_log"][hs].contiguous().cuda()
    outs = []
    for s in range(S):
        args = [d[n][s, :, hs].contiguous().cuda() for n in ("q", "k", "v", "z", "beta")]
        outs.append(kda.recurrent_step(*args, b, a, st))
    o_dec = torch.stack(outs, 1).float().cpu()  # [N, S, H, D]
    seq = lambda n: torch.stack([d[n][s, :, hs] for s in range(S)], 1).reshape(N * S, H, *d[n].shape[3:]).contiguous()  # noqa: E731
    cu = torch.arange(0, N * S + 1, S, dtype=torch.int32)
    o_pf, fs_pf = kda.chunk_fwd(*(seq(n).cuda() for n in ("q", "k", "v", "z", "beta")), b, a,
                                cu_seqlens=cu.cuda(), initial_state=S0.cuda(), output_final_state=True)
    torch.cuda.synchronize()
    o_pf = o_pf.float().cpu().reshape(N, S, H, -1)
    for n in range(N):
        for h in range(H):
            assert rel_err(o_dec[n, :, h].numpy(), o_pf[n, :, h].numpy()) <= TOL_BF16
            assert rel_err(st[n, h].cpu().numpy(), fs_pf[n, h].cpu().numpy()) <= TOL_BF16


@pytest.mark.parametrize("T", [8192, 8192 + 37])
def test_split_sequence_state_pass(T):
    """Long sequences with few heads take the split-sequence state pass (segment summaries,
    fold, per-segment output); checked against the oracle like any other case."""
    w = syn.Workload("cp", H=2, d=128, dtype="bf16", seq_len=T, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = syn.make_prefill(w, seed=41)
    assert kda.chunk_fwd_kernel_count(T, 1, 2, 128, 128, torch.bfloat16, d["cu_seqlens"]) == 5
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16)


def test_split_sequence_varlen_mix():
    """Split state pass with sequences of very different lengths, one of them empty."""
    w = syn.Workload("cpv", H=2, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = _varlen(w, [8192, 100, 0, 3000, 5000, 64], seed=42)
    assert kda.chunk_fwd_kernel_count(sum(d["lengths"]), 6, 2, 128, 128, torch.bfloat16, d["cu_seqlens"]) == 5
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16)


def test_split_sequence_final_state_aliases_initial_state():
    w = syn.Workload("cpa", H=2, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = _varlen(w, [8192, 300], seed=43)
    assert kda.chunk_fwd_kernel_count(sum(d["lengths"]), 2, 2, 128, 128, torch.bfloat16, d["cu_seqlens"]) == 5
    st = d["initial_state"].cuda().contiguous()
    dev = "cuda"
    o, _ = kda.chunk_fwd(*(d[n].to(dev) for n in ("q", "k", "v", "z", "beta")), d["dt_bias"].to(dev),
                         d["A_log"].to(dev), cu_seqlens=d["cu_seqlens"].to(dev), cu_seqlens_host=d["cu_seqlens"],
                         initial_state=st, final_state=st)
    torch.cuda.synchronize()
    compare_prefill(d, o.float().cpu(), st.cpu(), oracle_prefill(d), TOL_BF16)


# ----------------------------------------------------------------------------- output epilogue (Eq. 6)

EPS = 1e-6


def _epilogue_ref(d, res, g, w):
    """Oracle: per (sequence, head), the recurrence's output followed by the Eq. 6 epilogue."""
    cu = [int(x) for x in d["cu_seqlens"]]
    out = {}
    for (n, h), (o_ref, S_ref) in res.items():
        gg = g[cu[n]:cu[n + 1], h].double().numpy()
        out[(n, h)] = (R.output_gate(o_ref, gg, w[h].double().numpy(), EPS), S_ref)
    return out


@pytest.mark.parametrize("dtype,dv", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 32), ("bf16", 256)])
def test_output_gate_standalone(dtype, dv):
    T, H = 301, 3
    o = syn.make_tokens(T, H, dv, dv, dtype, 31, z_std=1.0)[2] * 3.0
    g, w = syn.make_output_gate_inputs(T, H, dv, dtype, 32)
    ref = R.output_gate(o.double().numpy(), g.double().numpy(), w.double().numpy()[None], EPS)
    tol = TOL_BF16 if dtype == "bf16" else 1e-5
    y = kda.output_gate(o.cuda(), g.cuda(), w.cuda(), EPS).float().cpu()
    y_now = kda.output_gate(o.cuda(), g.cuda(), None, EPS).float().cpu()
    ref_now = R.output_gate(o.double().numpy(), g.double().numpy(), None, EPS)
    oc = o.cuda().contiguous()
    kda.output_gate(oc, g.cuda(), w.cuda(), EPS, out=oc)  # in place
    for h in range(H):
        assert rel_err(y[:, h].numpy(), ref[:, h]) <= tol
        assert rel_err(y_now[:, h].numpy(), ref_now[:, h]) <= tol
        assert rel_err(oc[:, h].float().cpu().numpy(), ref[:, h]) <= tol


def test_prefill_4k_with_output_epilogue():
    """The benchmark workload with the output epilogue requested through kda_chunk_fwd."""
    d = syn.make_prefill(syn.PREFILL_4K, seed=1)
    g, w = syn.make_output_gate_inputs(4096, 32, 128, "bf16", 33)
    o, fs = run_prefill(d, out_gate=g.cuda(), out_norm_weight=w.cuda(), out_norm_eps=EPS)
    compare_prefill(d, o, fs, _epilogue_ref(d, oracle_prefill(d), g, w), TOL_BF16)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_varlen_ragged_with_output_epilogue(dtype, D):
    """Ragged lengths (empty, 1, chunk +-1, tails), tensor-core and fp32 paths, with the epilogue."""
    w_ = syn.Workload("ve", H=3, d=D, dtype=dtype, seq_len=None, z_std=1.5, b_range=1.0,
                      alog_std=0.25, s0_std=0.02)
    d = _varlen(w_, [1, 63, 64, 0, 65, 130, 200, 7], seed=24)
    T = sum(d["lengths"])
    g, w = syn.make_output_gate_inputs(T, 3, D, dtype, 34)
    o, fs = run_prefill(d, out_gate=g.cuda(), out_norm_weight=w.cuda(), out_norm_eps=EPS)
    compare_prefill(d, o, fs, _epilogue_ref(d, oracle_prefill(d), g, w),
                    TOL_F32 if dtype == "f32" else TOL_BF16)


def test_epilogue_through_prefill_equals_separate_call():
    """kda_chunk_fwd with out_gate == plain kda_chunk_fwd followed by kda_output_gate."""
    w_ = syn.Workload("fe", H=4, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0,
                      alog_std=0.25, s0_std=0.02)
    d = _varlen(w_, [700, 64, 333], seed=25)
    T = sum(d["lengths"])
    g, w = syn.make_output_gate_inputs(T, 4, 128, "bf16", 35)
    o_f, _ = run_prefill(d, out_gate=g.cuda(), out_norm_weight=w.cuda(), out_norm_eps=EPS)
    o_p, _ = run_prefill(d)
    o_s = kda.output_gate(o_p.to(torch.bfloat16).cuda(), g.cuda(), w.cuda(), EPS).float().cpu()
    for h in range(4):
        assert rel_err(o_f[:, h].numpy(), o_s[:, h].numpy()) <= 1e-6


# ----------------------------------------------------------------------------- speculative replay (section 5.4)

def _replay_inputs(D, dtype, N, H, Rw, M, seed):
    w = syn.Workload("rp", H=H, d=D, dtype=dtype, n_seq=N, seq_len=1, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02, decode_steps=Rw + M)
    d = syn.make_decode(w, seed=seed)
    win = lambda name, a, b: d[name][a:b].transpose(0, 1).contiguous()  # noqa: E731  [N, L, H, ...]
    cached = tuple(win(n, 0, Rw) for n in ("q", "k", "z", "v", "beta"))
    new = tuple(win(n, Rw, Rw + M) for n in ("q", "k", "z", "v", "beta"))
    return d, cached, new


def _replay_oracle(d, cached, new, nr, nc, n, h):
    def tup(t):
        q, k, z, v, beta = (x[n, :, h].double().numpy() for x in t)
        g = R.gate(z, d["dt_bias"][h].double().numpy(), float(d["A_log"][h]), d["g_min"])
        return q, k, v, g, beta
    return R.replay(tup(cached), nr, tup(new), nc, d["state"][n, h].double().numpy())


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f32"), (128, "f32"), (64, "bf16")])
def test_recurrent_replay_matches_oracle(D, dtype):
    """Accepted cached drafts replayed, bonus and new drafts run; every replay / commit count from 0 to
    the window, permuted state slots with a spare slot left untouched."""
    N, H, Rw, M = 6, 3, 4, 3
    d, cached, new = _replay_inputs(D, dtype, N, H, Rw, M, seed=13)
    nr = torch.tensor([0, 4, 2, 1, 3, 4], dtype=torch.int32)
    nc = torch.tensor([1, 0, 3, 1, 2, 1], dtype=torch.int32)
    slots = torch.tensor([5, 0, 3, 1, 2, 6], dtype=torch.int32)
    pool = torch.randn((7, H, D, D)) * 0.02
    pool[slots.long()] = d["state"]
    pool_gpu = pool.cuda()
    o = kda.recurrent_replay(tuple(x.cuda() for x in cached), nr.cuda(), tuple(x.cuda() for x in new), nc.cuda(),
                             d["dt_bias"].cuda(), d["A_log"].cuda(), pool_gpu, state_indices=slots.cuda())
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    out = pool_gpu.cpu()
    for n in range(N):
        for h in range(H):
            o_ref, S_ref = _replay_oracle(d, cached, new, int(nr[n]), int(nc[n]), n, h)
            assert rel_err(o[n, :, h].float().cpu().numpy(), o_ref) <= tol, (n, h)
            assert rel_err(out[int(slots[n]), h].numpy(), S_ref) <= tol, (n, h)
    assert torch.equal(out[4], pool[4])  # spare slot untouched


def test_recurrent_replay_equals_single_steps():
    """Replaying the accepted drafts and committing the bonus token leaves the state that one decode
    step per token would leave; the new tokens' outputs are those of continued single steps."""
    D, N, H, Rw, M = 128, 4, 2, 3, 4
    d, cached, new = _replay_inputs(D, "bf16", N, H, Rw, M, seed=14)
    nr = torch.full((N,), Rw, dtype=torch.int32)
    nc = torch.ones((N,), dtype=torch.int32)
    st_r = d["state"].clone().cuda()
    o_r = kda.recurrent_replay(tuple(x.cuda() for x in cached), nr.cuda(), tuple(x.cuda() for x in new),
                               nc.cuda(), d["dt_bias"].cuda(), d["A_log"].cuda(), st_r)
    st_s = d["state"].clone().cuda()
    outs = []
    for s in range(Rw + M):
        args = [d[n][s].contiguous().cuda() for n in ("q", "k", "v", "z", "beta")]
        outs.append(kda.recurrent_step(*args, d["dt_bias"].cuda(), d["A_log"].cuda(), st_s).float().cpu())
        if s == Rw:  # after the bonus token: the committed state
            st_commit = st_s.clone()
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    for n in range(N):
        for h in range(H):
            assert rel_err(st_r[n, h].cpu().numpy(), st_commit[n, h].cpu().numpy()) <= 1e-5
            o_steps = torch.stack([outs[Rw + j][n, h] for j in range(M)]).numpy()
            assert rel_err(o_r[n, :, h].float().cpu().numpy(), o_steps) <= 1e-2


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f32")])
def test_recurrent_replay_long_windows_many_states(D, dtype):
    """Windows of up to 19 tokens (several staging groups of 8) over more (sequence, head) states than
    the device keeps resident, so that each CTA runs several states back to back."""
    N, H, Rw, M = 48, 16, 10, 9
    d, cached, new = _replay_inputs(D, dtype, N, H, Rw, M, seed=16)
    g = torch.Generator().manual_seed(17)
    nr = torch.randint(0, Rw + 1, (N,), generator=g, dtype=torch.int32)
    nc = torch.randint(0, M + 1, (N,), generator=g, dtype=torch.int32)
    nr[0], nc[0], nr[1], nc[1] = Rw, M, 0, 0  # the longest window; nothing committed
    st = d["state"].clone().cuda()
    o = kda.recurrent_replay(tuple(x.cuda() for x in cached), nr.cuda(), tuple(x.cuda() for x in new), nc.cuda(),
                             d["dt_bias"].cuda(), d["A_log"].cuda(), st)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    out, o = st.cpu(), o.float().cpu()
    for n in range(N):
        for h in range(H):
            o_ref, S_ref = _replay_oracle(d, cached, new, int(nr[n]), int(nc[n]), n, h)
            assert rel_err(o[n, :, h].numpy(), o_ref) <= tol, (n, h)
            assert rel_err(out[n, h].numpy(), S_ref) <= tol, (n, h)


def test_recurrent_replay_bad_sequence_leaves_the_others_intact():
    """A sequence with an out-of-range count is skipped with KDA_ERR_BAD_TOKEN_COUNT; the states
    around it in the same launch are still computed."""
    D, N, H, Rw, M = 128, 40, 8, 3, 4
    d, cached, new = _replay_inputs(D, "bf16", N, H, Rw, M, seed=18)
    nr = torch.full((N,), 2, dtype=torch.int32)
    nc = torch.ones((N,), dtype=torch.int32)
    nr[17] = Rw + 1
    st = d["state"].clone().cuda()
    o = kda.recurrent_replay(tuple(x.cuda() for x in cached), nr.cuda(), tuple(x.cuda() for x in new), nc.cuda(),
                             d["dt_bias"].cuda(), d["A_log"].cuda(), st)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 11
    out, o = st.cpu(), o.float().cpu()
    assert torch.equal(out[17], d["state"][17])
    for n in (0, 16, 18, 39):
        for h in range(H):
            o_ref, S_ref = _replay_oracle(d, cached, new, int(nr[n]), int(nc[n]), n, h)
            assert rel_err(o[n, :, h].numpy(), o_ref) <= TOL_BF16, (n, h)
            assert rel_err(out[n, h].numpy(), S_ref) <= TOL_BF16, (n, h)


def test_recurrent_replay_nothing_committed_and_bad_counts():
    D, N, H = 64, 2, 2
    d, cached, new = _replay_inputs(D, "f32", N, H, 2, 2, seed=15)
    st = d["state"].clone().cuda()
    kda.recurrent_replay(tuple(x.cuda() for x in cached), torch.zeros(N, dtype=torch.int32, device="cuda"),
                         tuple(x.cuda() for x in new), torch.zeros(N, dtype=torch.int32, device="cuda"),
                         d["dt_bias"].cuda(), d["A_log"].cuda(), st)
    assert kda.get_device_error() == 0
    assert torch.equal(st.cpu(), d["state"])  # nothing replayed or committed: untouched
    kda.recurrent_replay(tuple(x.cuda() for x in cached), torch.tensor([0, 3], dtype=torch.int32, device="cuda"),
                         tuple(x.cuda() for x in new), torch.zeros(N, dtype=torch.int32, device="cuda"),
                         d["dt_bias"].cuda(), d["A_log"].cuda(), st)
    assert kda.get_device_error() == 11


# ----------------------------------------------------------------------------- failure detection

def test_bounded_wait_gives_up_and_context_stays_usable():
    """A wait nothing completes (an mbarrier with no arrival, through the bounded wait the kernels
    use) returns after about a second with KDA_ERR_DEVICE_TIMEOUT; the next call runs normally."""
    code, secs = kda.selftest_bounded_wait()
    assert code == 10  # KDA_ERR_DEVICE_TIMEOUT
    assert 0.5 <= secs <= 10.0, secs
    assert kda.get_device_error() == 0  # read and cleared
    d = syn.make_prefill(syn.TINY_F32, seed=0)
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_F32)


def test_captured_graph_replays_with_new_inputs():
    """kda_chunk_fwd captured in a CUDA graph, then replayed twice with new contents written into the
    same input buffers: each replay must match the oracle on its own inputs.  Uncaptured, this
    workload takes the fused schedule, whose packet flags carry a per-call host counter; the
    captured call must not depend on it (it runs the flag-free kernels)."""
    w = syn.PREFILL_4K
    ds = [syn.make_prefill(w, seed=s) for s in (11, 12)]
    T, H, D = sum(ds[0]["lengths"]), w.H, w.d
    cu_host = ds[0]["cu_seqlens"]
    assert kda.chunk_fwd_schedule(T, 1, H, D, D, torch.bfloat16, cu_host)["fused"]
    names = ("q", "k", "v", "z", "beta", "dt_bias", "A_log")
    buf = {n: ds[0][n].cuda() for n in names}
    cu = cu_host.cuda()
    o = torch.empty_like(buf["v"])
    fs = torch.empty((1, H, D, D), dtype=torch.float32, device="cuda")
    ws = torch.empty((kda.chunk_fwd_workspace_size(T, 1, H, D, D, torch.bfloat16, 64, cu_host),),
                     dtype=torch.uint8, device="cuda")

    def call():
        kda.chunk_fwd(*(buf[n] for n in names), g_min=ds[0]["g_min"], scale=ds[0]["scale"], cu_seqlens=cu,
                      cu_seqlens_host=cu_host, final_state=fs, workspace=ws, out=o)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for d in ds + ds[:1]:
        for n in names:
            buf[n].copy_(d[n])
        graph.replay()
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        worst = compare_prefill(d, o.float().cpu(), fs.cpu(), oracle_prefill(d, heads=None), TOL_BF16)
        assert worst < TOL_BF16


def test_debug_checks_report_non_finite_outputs():
    """kda_set_debug_checks(KDA_CHECK_FINITE): a NaN in one value vector reaches that head's outputs
    and state, and the check pass reports KDA_ERR_NUMERIC; clean inputs report nothing, and with the
    checks off nothing is reported either."""
    w = syn.Workload("dbg", H=2, d=64, dtype="f32", n_seq=1, seq_len=100, z_std=1.5, b_range=1.0,
                     alog_std=0.25)
    d = syn.make_prefill(w, seed=61)
    try:
        kda.set_debug_checks(kda.CHECK_FINITE)
        run_prefill(d)  # asserts no device error
        d["v"][37, 1, 5] = float("nan")
        o, fs = kda.chunk_fwd(*(d[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log")),
                              cu_seqlens=d["cu_seqlens"].cuda(), output_final_state=True)
        assert kda.get_device_error() == 12  # KDA_ERR_NUMERIC
        assert not torch.isfinite(fs[0, 1]).all() and torch.isfinite(fs[0, 0]).all()
        st = torch.zeros((3, 2, 64, 64), device="cuda")
        tok = lambda: torch.randn((3, 2, 64), device="cuda")  # noqa: E731
        kda.recurrent_step(tok(), tok(), tok(), tok(), torch.rand((3, 2), device="cuda"), None, None, st)
        assert kda.get_device_error() == 0
        st[1, 0, 3, 3] = float("inf")
        kda.recurrent_step(tok(), tok(), tok(), tok(), torch.rand((3, 2), device="cuda"), None, None, st)
        assert kda.get_device_error() == 12
    finally:
        kda.set_debug_checks(0)
    kda.chunk_fwd(*(d[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log")),
                  cu_seqlens=d["cu_seqlens"].cuda(), output_final_state=True)
    assert kda.get_device_error() == 0


@pytest.fixture
def team_schedule():
    """The chain-team launch runs only when asked for (the model never picks it)."""
    kda.set_chunk_schedule("team")
    yield
    kda.set_chunk_schedule("auto")


def _team_case(seed, lengths, H=8):
    w = syn.Workload("team", H=H, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    d = _varlen(w, lengths, seed=seed)
    sch = kda.chunk_fwd_schedule(sum(lengths), len(lengths), H, 128, 128, torch.bfloat16, d["cu_seqlens"])
    assert sch["team"] and sch["kernels"] == 1, sch
    return d


def test_team_schedule_varlen_with_states(team_schedule):
    """The chain-team launch (many chains: 20 sequences x 8 heads) on a ragged batch with empty,
    one-token, one-chunk and unaligned sequences and initial states: every (sequence, head) against
    the oracle; an empty sequence's final state is its initial state bit for bit."""
    rng = np.random.default_rng(71)
    lengths = [int(x) for x in rng.integers(0, 400, size=20)]
    lengths[3], lengths[7], lengths[11], lengths[15] = 0, 1, 64, 65
    d = _team_case(72, lengths)
    o, fs = run_prefill(d)
    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16)
    assert torch.equal(fs[3], d["initial_state"][3])


def test_team_schedule_final_state_aliases_initial_state(team_schedule):
    """In-place continuation under the chain-team launch: final_state is initial_state."""
    rng = np.random.default_rng(73)
    lengths = [int(x) for x in rng.integers(100, 700, size=24)]
    d = _team_case(74, lengths)
    ref = oracle_prefill(d)
    dev = "cuda"
    st = d["initial_state"].to(dev).clone()
    o, _ = kda.chunk_fwd(*(d[n].to(dev) for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log")),
                         cu_seqlens=d["cu_seqlens"].to(dev), cu_seqlens_host=d["cu_seqlens"],
                         initial_state=st, final_state=st)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    compare_prefill(d, o.float().cpu(), st.cpu(), ref, TOL_BF16)


def test_team_schedule_bad_cu_seqlens_reports_device_error(team_schedule):
    """The chain-team launch validates cu_seqlens in every CTA and runs nothing when it is inconsistent."""
    lengths = [100] * 20
    d = _team_case(75, lengths)
    cu = d["cu_seqlens"].clone()
    cu[6] = int(cu[5]) - 1  # no longer non-decreasing
    dev = "cuda"
    kda.chunk_fwd(*(d[n].to(dev) for n in ("q", "k", "v", "z", "beta")), None, None, cu_seqlens=cu.to(dev),
                  cu_seqlens_host=d["cu_seqlens"], output_final_state=True)
    assert kda.get_device_error() == 7


@pytest.mark.parametrize("schedule", ["separate", "team"])
def test_output_epilogue_inside_the_output_pass(schedule):
    """The epilogue applied by the output pass itself (separate kernels, chain teams) on a ragged batch
    with an empty sequence and states: per (sequence, head) against the oracle's recurrence followed by
    the Eq. 6 epilogue, and equal to the recurrence plus a separate kda_output_gate call."""
    w_ = syn.Workload("vi", H=8, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0,
                      alog_std=0.25, s0_std=0.02)
    rng = np.random.default_rng(81)
    lengths = [int(x) for x in rng.integers(0, 300, size=20)]
    lengths[2], lengths[9] = 0, 64
    d = _varlen(w_, lengths, seed=82)
    T = sum(lengths)
    g, w = syn.make_output_gate_inputs(T, 8, 128, "bf16", 83)
    try:
        kda.set_chunk_schedule(schedule)
        sch = kda.chunk_fwd_schedule(T, len(lengths), 8, 128, 128, torch.bfloat16, d["cu_seqlens"])
        assert sch[schedule] if schedule == "team" else not (sch["fused"] or sch["team"])
        o, fs = run_prefill(d, out_gate=g.cuda(), out_norm_weight=w.cuda(), out_norm_eps=EPS)
        o_plain, _ = run_prefill(d)
    finally:
        kda.set_chunk_schedule("auto")
    compare_prefill(d, o, fs, _epilogue_ref(d, oracle_prefill(d), g, w), TOL_BF16)
    y = kda.output_gate(o_plain.to(torch.bfloat16).cuda(), g.cuda(), w.cuda(), EPS).float().cpu()
    assert rel_err(o.numpy(), y.numpy()) <= 1e-2


@pytest.mark.parametrize("schedule", ["fused", "auto"])
def test_output_epilogue_on_long_chains(schedule):
    """The epilogue on long chains: T = 16421 tokens (a ragged last chunk), 4 heads, on the one-launch
    schedule (forced; the epilogue then runs as its own pass) and on the schedule the model picks for it
    (the split state pass: segment summaries, fold, output pass per segment applying the epilogue),
    against the oracle."""
    w_ = syn.Workload("lo", H=4, d=128, dtype="bf16", n_seq=1, seq_len=16421, z_std=1.5, b_range=1.0,
                      alog_std=0.25)
    d = syn.make_prefill(w_, seed=84)
    T = 16421
    g, w = syn.make_output_gate_inputs(T, 4, 128, "bf16", 85)
    try:
        kda.set_chunk_schedule(schedule)
        sch = kda.chunk_fwd_schedule(T, 1, 4, 128, 128, torch.bfloat16, d["cu_seqlens"])
        assert sch["fused"] if schedule == "fused" else sch["seg_len"] > 0
        assert sch["kernels"] == (1 if schedule == "fused" else 5)
        n_k = kda.chunk_fwd_kernel_count(T, 1, 4, 128, 128, torch.bfloat16, d["cu_seqlens"], out_gate=True)
        assert n_k == (2 if schedule == "fused" else 5)  # the one-launch schedule adds the epilogue pass
        o, fs = run_prefill(d, out_gate=g.cuda(), out_norm_weight=w.cuda(), out_norm_eps=EPS)
    finally:
        kda.set_chunk_schedule("auto")
    compare_prefill(d, o, fs, _epilogue_ref(d, oracle_prefill(d), g, w), TOL_BF16)


def test_shared_workspace_across_schedules_and_repeated_calls():
    """One workspace serves interleaved calls of different problems and schedules (separate kernels
    with the producers' item counter, the one-launch schedule with flags and counter, the split state
    pass with the output pass's unit counter), twelve times over: every call's result equals the
    first call of the same problem bit for bit, and the first ones match the oracle.  Counters and
    flags left in the workspace by one call (tagged with its own number, or reset by the planning
    kernel) never leak into the next."""
    w = syn.Workload("ws", H=4, d=128, dtype="bf16", seq_len=None, z_std=1.5, b_range=1.0, alog_std=0.25,
                     s0_std=0.02)
    rng = np.random.default_rng(97)
    cases = []
    for lengths, mode in (([int(x) for x in rng.integers(1, 700, size=12)], "separate"),
                          ([2000, 900], "fused"),
                          ([9000, 130], "auto")):
        d = _varlen(w, lengths, seed=int(rng.integers(1 << 20)))
        cases.append((d, mode))
    size = 0
    for d, mode in cases:
        kda.set_chunk_schedule(mode)
        try:
            size = max(size, kda.chunk_fwd_workspace_size(sum(d["lengths"]), len(d["lengths"]), 4, 128, 128,
                                                          torch.bfloat16, 64, d["cu_seqlens"]))
        finally:
            kda.set_chunk_schedule("auto")
    ws = torch.empty((size,), dtype=torch.uint8, device="cuda")
    first = {}
    try:
        for rep in range(12):
            for i, (d, mode) in enumerate(cases):
                kda.set_chunk_schedule(mode)
                o, fs = run_prefill(d, workspace=ws)
                if rep == 0:
                    first[i] = (o, fs)
                    compare_prefill(d, o, fs, oracle_prefill(d), TOL_BF16)
                else:
                    assert torch.equal(o, first[i][0]) and torch.equal(fs, first[i][1]), (rep, i, mode)
    finally:
        kda.set_chunk_schedule("auto")
    assert kda.get_device_error() == 0
