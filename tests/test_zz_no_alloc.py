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


def _compare(c, tol):
    fs_ref = torch.empty_like(c["s0"])
    o_ref, _ = kda.chunk_fwd(c["q"], c["k"], c["v"], c["z"], c["beta"], c["b"], c["a"],
                             cu_seqlens=c["cu"], initial_state=c["s0"], final_state=fs_ref)
    fs = torch.empty_like(c["s0"])
    o = torch.empty_like(o_ref)
    kda.chunk_fwd_static_ws(c["q"], c["k"], c["v"], c["z"], c["beta"], c["b"], c["a"], cu_seqlens=c["cu"],
                            cu_seqlens_host=c["cu_host"], initial_state=c["s0"], final_state=fs, out=o)
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
    # two calls in a row with different sizes and inputs: the buffer keeps the first call's bytes
    _compare(_case("bf16", 128, [200, 64, 1, 130], seed=31), TOL_BF16)
    _compare(_case("bf16", 128, [65, 300], seed=32), TOL_BF16)
    _compare(_case("f32", 64, [100, 7], seed=33), TOL_F32)


def test_static_workspace_rejects_oversized_problem(cuda_ok):
    L = kda.load_library()
    T, H = 1 << 15, 32  # far more scratch than the static buffer holds
    need = L.kda_chunk_fwd_workspace_size(T, 1, H, 128, 128, kda.KDA_BF16, 64, None)
    assert need > kda.STATIC_WORKSPACE_BYTES
    fake = 1 << 20  # never dereferenced: the size check fails before any launch
    a = kda.ChunkArgs(T=T, N=1, H=H, dk=128, dv=128, dtype=kda.KDA_BF16, q=fake, k=fake, z=fake,
                      v=fake, beta=fake, dt_bias=None, A_log=None, g_min=-5.0, scale=1.0,
                      cu_seqlens=None, cu_seqlens_host=None, initial_state=None, final_state=None,
                      o=fake + 4096, chunk_size=64)
    assert L.kda_chunk_fwd_static_ws(ctypes.byref(a), None) == 5  # KDA_ERR_WORKSPACE
