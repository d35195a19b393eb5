"""GPU parity of kda_chunk_bwd (backward of the chunked prefill) against exact fp64 gradients.

The reference is the fp64 reverse-mode derivative of the token recurrence of Eq. 1 with the gate
(``oracle.autograd_ref``), on the same inputs the kernel reads (bf16 inputs as rounded).  The loss
is sum(o * grad_o) + sum(S_T * grad_final_state).  Relative Frobenius error per (sequence, head)
for every gradient: 1e-4 for fp32 I/O, 1e-2 for bf16 I/O (gradients are stored in bf16).
"""
import numpy as np
import pytest
import torch

from linear_attention_kda_gb300 import kda, synthetic as syn
from oracle import autograd_ref as AG
from tests.gpu_util import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev(cuda_ok):
    torch.cuda.set_device(0)
    kda.load_library()


def _inputs(H, D, dtype, lengths, seed, with_s0=True, with_dst=True):
    T = sum(lengths)
    q, k, v, beta, z = syn.make_tokens(T, H, D, D, dtype, seed, z_std=1.5)
    b, a = syn.make_head_params(H, D, seed, b_range=1.0, alog_std=0.25)
    gen = torch.Generator().manual_seed(seed + 1000)
    d = dict(q=q, k=k, v=v, beta=beta, z=z, dt_bias=b, A_log=a, lengths=lengths,
             cu_seqlens=syn.cu_seqlens_of(lengths),
             S0=syn.make_state(len(lengths), H, D, D, 0.02, seed) if with_s0 else None,
             do=torch.randn((T, H, D), generator=gen).to(q.dtype),
             dST=(torch.randn((len(lengths), H, D, D), generator=gen) * 0.1) if with_dst else None)
    return d


def _run(d, gate, varlen=True):
    cu = d["cu_seqlens"].cuda() if varlen else None
    g = kda.chunk_bwd(*(d[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log", "do")),
                      cu_seqlens=cu, n_seq=len(d["lengths"]),
                      initial_state=None if d["S0"] is None else d["S0"].cuda(),
                      grad_final_state=None if d["dST"] is None else d["dST"].cuda(), gate=gate)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return {n: x.float().cpu().numpy() for n, x in g.items()}


def _ref(d, gate):
    f = lambda x: None if x is None else x.double().numpy()  # noqa: E731
    return AG.backward(f(d["q"]), f(d["k"]), f(d["v"]), f(d["z"]), f(d["beta"]), f(d["dt_bias"]), f(d["A_log"]),
                       d["cu_seqlens"], f(d["do"]), S0=f(d["S0"]), dST=f(d["dST"]), gate_kind=gate)


def _compare(d, got, ref, tol):
    cu = [int(x) for x in d["cu_seqlens"]]
    H = d["q"].shape[1]
    worst = {}
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        for h in range(H):
            pairs = [("initial_state", got["initial_state"][n, h], ref["dS0"][n, h])]
            if b > a:
                pairs += [(nm, got[nm][a:b, h], ref["d" + nm][a:b, h]) for nm in ("q", "k", "v", "z", "beta")]
            for nm, x, r in pairs:
                e = rel_err(x, r)
                assert np.isfinite(e) and e <= tol, f"d{nm} (seq {n}, head {h}): rel err {e:.3g} > {tol}"
                worst[nm] = max(worst.get(nm, 0.0), e)
    # the shared gate parameters, per head, each a sum over every token of every sequence
    sb, sa = gate_param_scales(ref["dz"], d["z"], d["dt_bias"], d["A_log"], d.get("gate", "lower_bound"))
    for h in range(H):
        eb = float(np.linalg.norm(got["dt_bias"][h] - ref["ddt_bias"][h])) / float(np.linalg.norm(sb[h]))
        ea = abs(float(got["A_log"][h]) - float(ref["dA_log"][h])) / float(sa[h])
        assert eb <= tol, f"d dt_bias (head {h}): error {eb:.3g} of the terms' magnitude > {tol}"
        assert ea <= tol, f"d A_log (head {h}): error {ea:.3g} of the terms' magnitude > {tol}"
        worst["dt_bias"] = max(worst.get("dt_bias", 0.0), eb)
        worst["A_log"] = max(worst.get("A_log", 0.0), ea)
    return worst


def gate_param_scales(dz, z, dt_bias, A_log, gate):
    """Magnitudes against which the dt_bias and A_log gradients of each head are measured.

    Both gates are functions of x = z + b, so d/db = sum_t dz_t exactly, and d/dA_log = sum_t,c dz w
    with w = z + b for Eq. 5 (g = g_min Sigmoid(e^A x): dg/dA = x dg/dz) and w = Softplus(x) / Sigmoid(x)
    for the softplus gate (g = -e^A Softplus(x): dg/dA = g, dg/dz = -e^A Sigmoid(x)).  These sums can
    cancel to a tiny fraction of their terms (a ratio near 3000 occurs in the fp32 varlen case), and
    a cancelling sum has no meaningful relative error of its own: its error is bounded by the
    tolerance times the sum of the terms' magnitudes.  Returns ([H, d_k] per-channel sum_t |dz|,
    [H] sum_t,c |dz w|) from the fp64 reference dz."""
    f = lambda t: t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)  # noqa: E731
    dz = f(dz)
    x = f(z) + f(dt_bias)[None]
    if gate == "softplus":
        w = np.logaddexp(0.0, x) * (1.0 + np.exp(-x))
    else:
        w = x
    return np.abs(dz).sum(0), np.abs(dz * w).sum((0, 2))


@pytest.mark.parametrize("gate", ["lower_bound", "softplus"])
def test_chunk_bwd_f32_varlen_matches_exact_gradients(gate):
    """Ragged batch (1, 63, 64, 65, 130 and an empty sequence) with initial and final state gradients."""
    d = _inputs(2, 64, "f32", [1, 63, 64, 65, 130, 0], seed=51)
    d["gate"] = gate
    _compare(d, _run(d, gate), _ref(d, gate), TOL_F32)


def test_chunk_bwd_bf16_d128_matches_exact_gradients():
    d = _inputs(2, 128, "bf16", [200, 77], seed=52)
    _compare(d, _run(d, "lower_bound"), _ref(d, "lower_bound"), TOL_BF16)


def test_chunk_bwd_bf16_d128_ragged_with_empty_sequence():
    """The tensor-core chains and value side on a ragged bf16 batch: an empty sequence (no chunks:
    d initial_state is d final_state passed through), one token, exactly one chunk, a chunk and one
    token, and two and a half chunks."""
    d = _inputs(2, 128, "bf16", [0, 1, 64, 65, 160], seed=57)
    _compare(d, _run(d, "lower_bound"), _ref(d, "lower_bound"), TOL_BF16)


def test_chunk_bwd_f32_d128_equal_lengths_without_states():
    """Two sequences of 96 tokens given by N alone (no cu_seqlens), zero initial state, no final-state
    gradient: d initial_state is then the full adjoint of the state entering each sequence."""
    d = _inputs(3, 128, "f32", [96, 96], seed=53, with_s0=False, with_dst=False)
    _compare(d, _run(d, "lower_bound", varlen=False), _ref(d, "lower_bound"), TOL_F32)


def test_chunk_bwd_optional_outputs_skipped():
    d = _inputs(1, 64, "f32", [70], seed=54)
    g = kda.chunk_bwd(*(d[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log", "do")),
                      cu_seqlens=d["cu_seqlens"].cuda(), initial_state=d["S0"].cuda(), param_grads=False,
                      state_grad=False)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert set(g) == {"q", "k", "v", "z", "beta"}
    ref = _ref(dict(d, dST=None), "lower_bound")
    assert rel_err(g["q"].cpu().numpy()[:, 0], ref["dq"][:, 0]) <= TOL_F32


def test_chunk_bwd_full_prefill_workload_sampled_heads():
    """The benchmark's workload (T = 4096, H = 32, d = 128, bf16) with the bench's launch: every
    gradient of two sampled heads (first and last) against exact fp64 gradients of the full sequence."""
    w = syn.PREFILL_4K
    dd = syn.make_prefill(w, seed=1)
    T, H = dd["q"].shape[0], w.H
    gen = torch.Generator().manual_seed(78)
    do = torch.randn((T, H, w.d), generator=gen).to(torch.bfloat16)
    dST = torch.randn((1, H, w.d, w.d), generator=gen) * 0.1
    g = kda.chunk_bwd(*(dd[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log")), do.cuda(),
                      cu_seqlens=dd["cu_seqlens"].cuda(), grad_final_state=dST.cuda())
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    got = {n: x.float().cpu().numpy() for n, x in g.items()}
    f = lambda x: x.double().numpy()  # noqa: E731
    for h in (0, H - 1):
        r = AG.head_backward(f(dd["q"][:, h]), f(dd["k"][:, h]), f(dd["v"][:, h]), f(dd["z"][:, h]),
                             f(dd["beta"][:, h]), f(dd["dt_bias"][h]), float(dd["A_log"][h]), None,
                             f(do[:, h]), f(dST[0, h]))
        for nm in ("q", "k", "v", "z", "beta"):
            assert rel_err(got[nm][:, h], r["d" + nm]) <= TOL_BF16, (nm, h)
        assert rel_err(got["initial_state"][0, h], r["dS0"]) <= TOL_BF16, h
        sb, sa = gate_param_scales(r["dz"][:, None], f(dd["z"][:, h])[:, None], f(dd["dt_bias"][h])[None],
                                   None, "lower_bound")
        assert np.linalg.norm(got["dt_bias"][h] - r["db"]) <= TOL_BF16 * np.linalg.norm(sb[0]), h
        assert abs(got["A_log"][h] - r["dA_log"]) <= TOL_BF16 * sa[0], h


def test_chunk_bwd_empty_batch():
    """T = 0 over two sequences, through the C ABI with NaN-filled gradient buffers.
    - Eq. 1 takes no step, so S_T = S_0.
    - d initial_state is then d final_state bit for bit, or zeros without it.
    - The dt_bias and A_log gradients are zero and are written as such."""
    import ctypes
    H, D, N = 2, 64, 2
    L = kda.load_library()
    b, a = (x.cuda() for x in syn.make_head_params(H, D, 4, b_range=1.0, alog_std=0.25))
    dST = (torch.randn((N, H, D, D), generator=torch.Generator().manual_seed(5)) * 0.1).cuda()
    cu = torch.zeros(N + 1, dtype=torch.int32, device="cuda")
    need = int(L.kda_chunk_bwd_workspace_size(0, N, H, D, D, 64))
    ws = torch.empty((max(need, 1),), dtype=torch.uint8, device="cuda")
    for with_dst in (True, False):
        nan = float("nan")
        gdb = torch.full((H, D), nan, device="cuda")
        gda = torch.full((H,), nan, device="cuda")
        gS0 = torch.full((N, H, D, D), nan, device="cuda")
        args = kda.ChunkBwdArgs(T=0, N=N, H=H, dk=D, dv=D, dtype=kda.KDA_F32, dt_bias=b.data_ptr(),
                                A_log=a.data_ptr(), g_min=-5.0, scale=1.0, cu_seqlens=cu.data_ptr(),
                                grad_final_state=dST.data_ptr() if with_dst else None,
                                grad_dt_bias=gdb.data_ptr(), grad_A_log=gda.data_ptr(),
                                grad_initial_state=gS0.data_ptr(), chunk_size=64, gate_kind=0)
        assert L.kda_chunk_bwd(ctypes.byref(args), ws.data_ptr(), ws.numel(), None) == 0
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        assert torch.equal(gS0, dST) if with_dst else torch.count_nonzero(gS0.nan_to_num(1.0)).item() == 0
        assert torch.count_nonzero(gdb.nan_to_num(1.0)).item() == 0
        assert torch.count_nonzero(gda.nan_to_num(1.0)).item() == 0


@pytest.mark.parametrize("gate,dtype,D", [("lower_bound", "f32", 64), ("softplus", "f32", 64),
                                           ("lower_bound", "bf16", 128)])
def test_chunk_bwd_segmented_long_sequence(gate, dtype, D):
    """One sequence given less workspace than the one-pass size runs in segments (here the minimum:
    segments of 16 chunks, so T = 2 x 1024 + 300 tokens makes three, the last ragged): every gradient
    against the exact fp64 gradients (1e-4 for fp32, 1e-2 for bf16 I/O, with S0 and dS_T), and equal to
    the one-pass result but for the rounding of the per-segment sums of the dt_bias and A_log gradients."""
    d = _inputs(2, D, dtype, [2 * 1024 + 300], 91)
    d["gate"] = gate
    T, H, D = d["q"].shape
    full = kda.chunk_bwd_workspace_size(T, 1, H, D, D)
    small = kda.chunk_bwd_workspace_size(T, 1, H, D, D, minimum=True)
    assert 0 < small < full
    dev = {n: d[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log", "do")}
    args = [dev[n] for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log", "do")]
    kw = dict(initial_state=d["S0"].cuda(), grad_final_state=d["dST"].cuda(), gate=gate)
    # workspaces full of NaN: no gradient may depend on scratch the call did not write
    seg = kda.chunk_bwd(*args, workspace=torch.full((small,), 0xFF, dtype=torch.uint8, device="cuda"), **kw)
    one = kda.chunk_bwd(*args, workspace=torch.full((full,), 0xFF, dtype=torch.uint8, device="cuda"), **kw)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    seg = {n: x.float().cpu().numpy() for n, x in seg.items()}
    one = {n: x.float().cpu().numpy() for n, x in one.items()}
    _compare(d, seg, _ref(d, gate), TOL_F32 if dtype == "f32" else TOL_BF16)
    for n in ("q", "k", "v", "z", "beta", "initial_state"):  # the same arithmetic, bf16 rounding aside
        assert rel_err(seg[n], one[n]) <= (1e-6 if dtype == "f32" else 4e-3), n
    for n in ("dt_bias", "A_log"):
        assert np.allclose(seg[n], one[n], rtol=1e-4, atol=1e-5 * float(np.abs(one[n]).max())), n


def test_chunk_bwd_workspace_too_small_or_batched():
    """Below the minimum the call is refused; a batch of several sequences needs the one-pass size."""
    d = _inputs(2, 64, "f32", [1500, 900], 93)
    T, H, D = d["q"].shape
    full = kda.chunk_bwd_workspace_size(T, 2, H, D, D)
    assert kda.chunk_bwd_workspace_size(T, 2, H, D, D, minimum=True) == full
    args = [d[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log", "do")]
    with pytest.raises(kda.KDAError, match="KDA_ERR_WORKSPACE"):
        kda.chunk_bwd(*args, cu_seqlens=d["cu_seqlens"].cuda(),
                      workspace=torch.empty((full - 256,), dtype=torch.uint8, device="cuda"))
    small = kda.chunk_bwd_workspace_size(2400, 1, H, D, D, minimum=True)
    a1 = [x[:2400] if x.dim() >= 2 and x.shape[0] == T else x for x in args]
    with pytest.raises(kda.KDAError, match="KDA_ERR_WORKSPACE"):
        kda.chunk_bwd(*a1, workspace=torch.empty((small - 256,), dtype=torch.uint8, device="cuda"))


def test_chunk_bwd_varlen_ignores_stale_workspace():
    """A varlen batch's chunk-slot bound exceeds its chunks; the slots past the last chunk must not
    reach the dt_bias and A_log sums: the pass on a workspace full of NaN equals the exact gradients."""
    d = _inputs(2, 64, "f32", [1, 63, 64, 65, 130, 0, 7], 95)
    T, H, D = d["q"].shape
    ws = torch.full((kda.chunk_bwd_workspace_size(T, 7, H, D, D),), 0xFF, dtype=torch.uint8, device="cuda")
    g = kda.chunk_bwd(*(d[n].cuda() for n in ("q", "k", "v", "z", "beta", "dt_bias", "A_log", "do")),
                      cu_seqlens=d["cu_seqlens"].cuda(), initial_state=d["S0"].cuda(),
                      grad_final_state=d["dST"].cuda(), workspace=ws)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    _compare(d, {n: x.float().cpu().numpy() for n, x in g.items()}, _ref(d, "lower_bound"), TOL_F32)
