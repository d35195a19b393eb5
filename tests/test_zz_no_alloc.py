"""kda_chunk_fwd_static_ws: prefill for callers that cannot allocate device memory.

Callers such as engine plugins (which receive only input/output pointers while
the engine owns all other device memory) cannot hand the library a scratch
workspace.  This entry point uses a fixed scratch buffer inside the library
instead.  The test calls it through the C ABI twice in a row, on different
inputs, and checks each result against kda_chunk_fwd (caller workspace) on
the same inputs -- so stale contents left by the first call cannot leak into
the second.  It also checks that a problem too large for the buffer is refused
before any launch.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from linear_attention_kda_gb300 import kda, synthetic as syn
from tests.gpu_util import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu


def _case(dtype, D, lengths, seed):
    w = syn.Workload("na", H=3, d=D, dtype=dtype, seq_len=None, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
    T = sum(lengths)
    q, k, v, beta, z = syn.make_tokens(T, w.H, D, D, dtype, seed, z_std=w.z_std)
    b, a = syn.make_head_params(w.H, D, seed, b_range=1.0, alog_std=0.25)
    s0 = syn.make_state(len(lengths), w.H, D, D, 0.02, seed)
    cu = syn.cu_seqlens_of(lengths)
    dev = "cuda"
    return dict(q=q.to(dev), k=k.to(dev), v=v.to(dev), z=z.to(dev), beta=beta.to(dev), b=b.to(dev),
                a=a.to(dev), s0=s0.to(dev), cu=cu.to(dev), cu_host=cu, H=w.H, N=len(lengths))


def _compare(c, tol, gate="lower_bound"):
    fs_ref = torch.empty_like(c["s0"])
    o_ref, _ = kda.chunk_fwd(c["q"], c["k"], c["v"], c["z"], c["beta"], c["b"], c["a"],
                             cu_seqlens=c["cu"], initial_state=c["s0"], final_state=fs_ref, gate=gate)
    fs = torch.empty_like(c["s0"])
    o = torch.empty_like(o_ref)
    kda.chunk_fwd_static_ws(c["q"], c["k"], c["v"], c["z"], c["beta"], c["b"], c["a"], cu_seqlens=c["cu"],
                            cu_seqlens_host=c["cu_host"], initial_state=c["s0"], final_state=fs, out=o, gate=gate)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(fs).all()
    cu = [int(x) for x in c["cu_host"]]
    for n in range(c["N"]):
        for h in range(c["H"]):
            a, b = cu[n], cu[n + 1]
            if b > a:
                assert rel_err(o[a:b, h].float().cpu().numpy(), o_ref[a:b, h].float().cpu().numpy()) <= tol
            assert rel_err(fs[n, h].cpu().numpy(), fs_ref[n, h].cpu().numpy()) <= tol


def test_static_workspace_matches_caller_workspace_twice(cuda_ok):
    torch.cuda.set_device(0)
    kda.load_library()
    # calls in a row with different sizes and inputs: the buffer keeps the previous call's bytes
    _compare(_case("bf16", 128, [200, 64, 1, 130], seed=31), TOL_BF16)
    _compare(_case("bf16", 128, [65, 300], seed=32), TOL_BF16)
    _compare(_case("f32", 64, [100, 7], seed=33), TOL_F32)
    # the unbounded softplus gate takes the fp32 path, whose scratch is sized separately
    _compare(_case("bf16", 128, [129, 40], seed=34), TOL_BF16, gate="softplus")


def test_static_workspace_rejects_oversized_problem(cuda_ok):
    """A problem just too large for the buffer (T = 4096, H = 32, bf16, d = 128: about 146 MiB of
    scratch) is refused before anything runs.  Every pointer is a real device tensor, so even a
    regressed size check could only compute, never touch memory it does not own."""
    L = kda.load_library()
    T, H, D = 4096, 32, 128
    need = L.kda_chunk_fwd_workspace_size(T, 1, H, D, D, kda.KDA_BF16, 64, None)
    assert need > kda.STATIC_WORKSPACE_BYTES
    q, k, v, z = (torch.zeros((T, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(4))
    beta = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    o = torch.full((T, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    a = kda.ChunkArgs(T=T, N=1, H=H, dk=D, dv=D, dtype=kda.KDA_BF16, q=q.data_ptr(), k=k.data_ptr(),
                      z=z.data_ptr(), v=v.data_ptr(), beta=beta.data_ptr(), dt_bias=None, A_log=None, g_min=-5.0,
                      scale=1.0, cu_seqlens=None, cu_seqlens_host=None, initial_state=None, final_state=None,
                      o=o.data_ptr(), chunk_size=64)
    assert L.kda_chunk_fwd_static_ws(ctypes.byref(a), None) == 5  # KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o.float() == 7.0).all())  # nothing ran
    # the softplus gate's fp32-path scratch is larger: a size that fits the bounded gate is refused
    T2, H2 = 4096, 10
    need_b = L.kda_chunk_fwd_workspace_size_gate(T2, 1, H2, D, D, kda.KDA_BF16, 64, None, 0)
    need_s = L.kda_chunk_fwd_workspace_size_gate(T2, 1, H2, D, D, kda.KDA_BF16, 64, None, 1)
    assert need_b <= kda.STATIC_WORKSPACE_BYTES < need_s
    a2 = kda.ChunkArgs(T=T2, N=1, H=H2, dk=D, dv=D, dtype=kda.KDA_BF16, q=q.data_ptr(), k=k.data_ptr(),
                       z=z.data_ptr(), v=v.data_ptr(), beta=beta.data_ptr(), dt_bias=None, A_log=None, g_min=-5.0,
                       scale=1.0, cu_seqlens=None, cu_seqlens_host=None, initial_state=None, final_state=None,
                       o=o.data_ptr(), chunk_size=64, gate_kind=1)
    assert L.kda_chunk_fwd_static_ws(ctypes.byref(a2), None) == 5
    # so is the bounded gate below g_min = -5.5, which runs on the same fp32 path
    a2.gate_kind, a2.g_min = 0, -8.0
    assert L.kda_chunk_fwd_static_ws(ctypes.byref(a2), None) == 5
    torch.cuda.synchronize()
    assert bool((o.float() == 7.0).all())
