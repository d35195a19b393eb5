"""Host-only checks of the C ABI (no GPU needed, no kernel launched).

* libkda.so loads and exports every function include/kda.h declares.
* The ctypes mirrors of the argument structs match the C layout (checked by
  compiling a small C program against include/kda.h with gcc).
* Host validation rejects bad arguments with the documented status before any
  launch: only cases that fail validation are sent through the ABI here, so no
  fake pointer ever reaches a kernel.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
import torch

from linear_attention_kda_gb300 import build as kbuild, kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(kda_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"kda_gate", "kda_chunk_fwd", "kda_recurrent_step"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libkda does not export {n}"
    assert set(kda.EXPORTED) <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", kbuild.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), f"{n} not a defined text symbol"


def test_abi_version_and_strings(lib):
    assert lib.kda_abi_version() == 5
    for code, name in kda._STATUS.items():
        s = lib.kda_status_string(code).decode()
        assert s and s != "unknown status", name
    assert lib.kda_status_string(999).decode() == "unknown status"


_LAYOUT_C = r"""
#include <stddef.h>
#include <stdio.h>
#include "kda.h"
#define F(S, f) printf(#S " " #f " %zu\n", offsetof(S, f));
int main(void) {
  printf("kda_gate_args sizeof %zu\n", sizeof(kda_gate_args));
  printf("kda_chunk_args sizeof %zu\n", sizeof(kda_chunk_args));
  printf("kda_step_args sizeof %zu\n", sizeof(kda_step_args));
  printf("kda_output_gate_args sizeof %zu\n", sizeof(kda_output_gate_args));
  printf("kda_replay_args sizeof %zu\n", sizeof(kda_replay_args));
  printf("kda_chunk_bwd_args sizeof %zu\n", sizeof(kda_chunk_bwd_args));
  %FIELDS%
  return 0;
}
"""


def test_struct_layout_matches_header(tmp_path):
    fields = []
    for cname, cls in (("kda_gate_args", kda.GateArgs), ("kda_chunk_args", kda.ChunkArgs),
                       ("kda_step_args", kda.StepArgs), ("kda_output_gate_args", kda.OutputGateArgs),
                       ("kda_replay_args", kda.ReplayArgs), ("kda_chunk_bwd_args", kda.ChunkBwdArgs)):
        for f, _ in cls._fields_:
            fields.append(f"F({cname}, {f})")
    src = tmp_path / "layout.c"
    src.write_text(_LAYOUT_C.replace("%FIELDS%", "\n  ".join(fields)))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {}
    for ln in lines:
        if ln.strip():
            s, f, v = ln.split()
            got[(s, f)] = int(v)
    for cname, cls in (("kda_gate_args", kda.GateArgs), ("kda_chunk_args", kda.ChunkArgs),
                       ("kda_step_args", kda.StepArgs), ("kda_output_gate_args", kda.OutputGateArgs),
                       ("kda_replay_args", kda.ReplayArgs), ("kda_chunk_bwd_args", kda.ChunkBwdArgs)):
        assert got[(cname, "sizeof")] == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert got[(cname, f)] == getattr(cls, f).offset, (cname, f)


FAKE = 1 << 20  # 16-byte aligned fake device address; never dereferenced (validation fails first)


def _chunk(**kw):
    base = dict(T=128, N=1, H=2, dk=128, dv=128, dtype=kda.KDA_BF16, q=FAKE, k=FAKE + 1024,
                z=FAKE + 2048, v=FAKE + 4096, beta=FAKE + 8192, dt_bias=None, A_log=None,
                g_min=-5.0, scale=1.0, cu_seqlens=None, cu_seqlens_host=None, initial_state=None,
                final_state=None, o=FAKE + 16384, chunk_size=64)
    base.update(kw)
    return kda.ChunkArgs(**base)


def _call_chunk(lib, a, ws=FAKE, ws_bytes=1 << 40):
    return lib.kda_chunk_fwd(ctypes.byref(a), ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=1 << 31), 2),           # token indices are 32-bit: T above INT32_MAX is refused
    (dict(dk=96, dv=96), 2),
    (dict(dk=128, dv=64), 2),
    (dict(chunk_size=32), 2),
    (dict(dtype=7), 3),
    (dict(N=0), 1),
    (dict(T=-1), 1),
    (dict(H=0), 1),
    (dict(g_min=0.0), 1),
    (dict(g_min=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(T=130, N=4), 1),          # equal-length split must divide T
    (dict(q=None), 1),
    (dict(o=FAKE), 1),              # o aliases q
    (dict(q=FAKE + 8), 4),
    (dict(o=FAKE + 16392), 4),
    (dict(initial_state=FAKE + 4), 4),
    (dict(out_gate=FAKE + 32768, out_norm_eps=0.0), 1),          # epilogue needs eps > 0
    (dict(out_gate=FAKE + 16384, out_norm_eps=1e-6), 1),         # gate aliases o
    (dict(out_gate=FAKE + 32776, out_norm_eps=1e-6), 4),
    (dict(out_gate=FAKE + 32768, out_norm_weight=FAKE + 40964, out_norm_eps=1e-6), 4),
    (dict(gate_kind=2), 1),                                      # no such gate
    (dict(gate_kind=-1), 1),
    (dict(gate_kind=1, g_min=0.0, q=None), 1),                   # softplus ignores g_min; q still checked
])
def test_chunk_fwd_rejects(lib, kw, code):
    assert _call_chunk(lib, _chunk(**kw)) == code


def test_chunk_fwd_workspace_checks(lib):
    a = _chunk()
    need = lib.kda_chunk_fwd_workspace_size(128, 1, 2, 128, 128, kda.KDA_BF16, 64, None)
    assert need > 0
    assert _call_chunk(lib, a, ws=None) == 5
    assert _call_chunk(lib, a, ws_bytes=need - 1) == 5
    assert _call_chunk(lib, a, ws=FAKE + 16, ws_bytes=need) == 4
    assert lib.kda_chunk_fwd_workspace_size(128, 1, 2, 96, 96, kda.KDA_BF16, 64, None) == 0
    assert lib.kda_chunk_fwd_workspace_size(128, 0, 2, 128, 128, kda.KDA_BF16, 64, None) == 0
    # the plain call is gate kind 0; the softplus gate takes the fp32 path, whose records are larger
    assert lib.kda_chunk_fwd_workspace_size_gate(128, 1, 2, 128, 128, kda.KDA_BF16, 64, None, 0) == need
    sp = lib.kda_chunk_fwd_workspace_size_gate(128, 1, 2, 128, 128, kda.KDA_BF16, 64, None, 1)
    assert sp > need
    assert sp == lib.kda_chunk_fwd_workspace_size(128, 1, 2, 128, 128, kda.KDA_F32, 64, None)
    assert lib.kda_chunk_fwd_workspace_size_gate(128, 1, 2, 128, 128, kda.KDA_BF16, 64, None, 3) == 0
    assert _call_chunk(lib, _chunk(gate_kind=1), ws_bytes=need) == 5
    # a bounded gate below g_min = -5.5 runs on the fp32 path (16 tokens of decay would leave fp32 range in
    # the tensor-core path's scaled images): it needs the fp32 path's workspace
    assert _call_chunk(lib, _chunk(g_min=-8.0), ws_bytes=need) == 5
    assert _call_chunk(lib, _chunk(g_min=-8.0), ws=FAKE + 16, ws_bytes=sp) == 4  # size accepted, then alignment
    assert _call_chunk(lib, _chunk(g_min=-5.5), ws=FAKE + 16, ws_bytes=need) == 4
    assert kda.chunk_fwd_schedule(4096, 1, 32, 128, 128, torch.bfloat16, g_min=-8.0)["kernels"] == 3
    assert kda.chunk_fwd_schedule(4096, 1, 32, 128, 128, torch.bfloat16, g_min=-5.0)["fused"]
    # the boundary: -5.5 itself stays on the tensor cores, the next float below it does not
    below = float(np.nextafter(np.float32(-5.5), np.float32(-6.0)))
    assert kda.chunk_fwd_schedule(4096, 1, 32, 128, 128, torch.bfloat16, g_min=-5.5)["fused"]
    assert kda.chunk_fwd_schedule(4096, 1, 32, 128, 128, torch.bfloat16, g_min=below)["kernels"] == 3
    assert kda.chunk_fwd_workspace_size(4096, 1, 32, 128, 128, torch.bfloat16, g_min=below) == \
        kda.chunk_fwd_workspace_size(4096, 1, 32, 128, 128, torch.bfloat16, gate="softplus")


def test_chunk_fwd_host_seqlens_validated(lib):
    cu = (ctypes.c_int32 * 3)(0, 100, 90)
    a = _chunk(T=90, N=2, cu_seqlens=FAKE + 32768, cu_seqlens_host=ctypes.addressof(cu))
    assert _call_chunk(lib, a) == 1
    cu2 = (ctypes.c_int32 * 3)(0, 50, 128)
    a = _chunk(T=100, N=2, cu_seqlens=FAKE + 32768, cu_seqlens_host=ctypes.addressof(cu2))
    assert _call_chunk(lib, a) == 1


def _step(**kw):
    base = dict(N=4, H=2, dk=128, dv=128, dtype=kda.KDA_BF16, q=FAKE, k=FAKE + 1024, z=FAKE + 2048,
                v=FAKE + 4096, beta=FAKE + 8192, dt_bias=None, A_log=None, g_min=-5.0, scale=1.0,
                state=FAKE + 65536, state_indices=None, num_slots=0, o=FAKE + 16384)
    base.update(kw)
    return kda.StepArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(N=1 << 30, H=4), 2),       # N x H above INT32_MAX
    (dict(dk=32, dv=32), 2),
    (dict(dtype=5), 3),
    (dict(H=0), 1),
    (dict(state=None), 1),
    (dict(num_slots=2), 1),        # fewer slots than sequences without an index map
    (dict(state=FAKE + 65544), 4),
    (dict(beta=FAKE + 8193), 4),
    (dict(g_min=1.0), 1),
    (dict(gate_kind=7), 1),
    (dict(gate_kind=1, g_min=1.0, state=None), 1),   # g_min ignored, the state still required
])
def test_recurrent_step_rejects(lib, kw, code):
    assert lib.kda_recurrent_step(ctypes.byref(_step(**kw)), None) == code


def test_gate_rejects(lib):
    a = kda.GateArgs(T=8, N=1, H=1, dk=16, dtype=kda.KDA_F32, z=FAKE, dt_bias=None, A_log=None,
                     g_min=-5.0, chunk_size=0, cu_seqlens=None, out=FAKE + 4096)
    a.g_min = 0.5
    assert lib.kda_gate(ctypes.byref(a), None) == 1
    a.g_min = -5.0
    a.z = FAKE + 2
    assert lib.kda_gate(ctypes.byref(a), None) == 4
    a.z = FAKE
    a.chunk_size = 4
    a.N = 3  # 8 tokens do not split into 3 equal sequences
    assert lib.kda_gate(ctypes.byref(a), None) == 1
    a.chunk_size = 1000
    assert lib.kda_gate(ctypes.byref(a), None) == 1
    a.chunk_size = 0
    a.N = 1
    a.gate_kind = 5
    assert lib.kda_gate(ctypes.byref(a), None) == 1
    a.gate_kind = 1
    a.g_min = 0.5  # ignored by the softplus gate: the call then fails only on the misaligned z
    a.z = FAKE + 2
    assert lib.kda_gate(ctypes.byref(a), None) == 4


def _og(**kw):
    base = dict(T=16, H=2, dv=128, dtype=kda.KDA_BF16, o=FAKE, g=FAKE + 8192, norm_weight=None, eps=1e-6,
                y=FAKE + 16384)
    base.update(kw)
    return kda.OutputGateArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(dv=96), 2),
    (dict(dtype=4), 3),
    (dict(H=0), 1),
    (dict(T=-1), 1),
    (dict(eps=0.0), 1),
    (dict(eps=float("nan")), 1),
    (dict(g=None), 1),
    (dict(y=FAKE + 8192), 1),       # y aliases g
    (dict(o=FAKE + 8), 4),
    (dict(norm_weight=FAKE + 32772), 4),
])
def test_output_gate_rejects(lib, kw, code):
    assert lib.kda_output_gate(ctypes.byref(_og(**kw)), None) == code


def _rp(**kw):
    base = dict(N=4, H=2, dk=128, dv=128, dtype=kda.KDA_BF16, R=3, rq=FAKE, rk=FAKE + 1024, rz=FAKE + 2048,
                rv=FAKE + 4096, rbeta=FAKE + 8192, n_replay=FAKE + 12288, M=2, q=FAKE + 16384, k=FAKE + 20480,
                z=FAKE + 24576, v=FAKE + 28672, beta=FAKE + 32768, n_commit=FAKE + 36864, dt_bias=None,
                A_log=None, g_min=-5.0, scale=1.0, state=FAKE + 65536, state_indices=None, num_slots=0,
                o=FAKE + 40960)
    base.update(kw)
    return kda.ReplayArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(N=1 << 20, M=1 << 10, H=4), 2),   # N x window x H above INT32_MAX
    (dict(dk=96, dv=96), 2),
    (dict(dtype=5), 3),
    (dict(M=0), 1),
    (dict(R=-1), 1),
    (dict(n_commit=None), 1),
    (dict(n_replay=None), 1),        # R > 0 needs the replay counts
    (dict(rq=None), 1),
    (dict(state=FAKE + 65544), 4),
    (dict(rq=FAKE + 8), 4),
    (dict(n_commit=FAKE + 36866), 4),
    (dict(g_min=1.0), 1),
    (dict(gate_kind=2), 1),
])
def test_recurrent_replay_rejects(lib, kw, code):
    assert lib.kda_recurrent_replay(ctypes.byref(_rp(**kw)), None) == code


def test_empty_inputs_are_noops(lib):
    # T = 0 gate / N = 0 decode return KDA_OK before touching any pointer or the device
    a = kda.GateArgs(T=0, N=1, H=1, dk=16, dtype=kda.KDA_F32, z=None, dt_bias=None, A_log=None,
                     g_min=-5.0, chunk_size=0, cu_seqlens=None, out=None)
    assert lib.kda_gate(ctypes.byref(a), None) == 0
    assert lib.kda_recurrent_step(ctypes.byref(_step(N=0, q=None)), None) == 0
    assert lib.kda_output_gate(ctypes.byref(_og(T=0, o=None, g=None, y=None)), None) == 0
    assert lib.kda_recurrent_replay(ctypes.byref(_rp(N=0, q=None)), None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_args_stop_at_device_check_without_gpu(lib):
    # Passes validation, then finds no sm_103 device: nothing is launched.
    assert _call_chunk(lib, _chunk()) == 9
    assert lib.kda_recurrent_step(ctypes.byref(_step()), None) == 9
    assert lib.kda_output_gate(ctypes.byref(_og()), None) == 9
    assert lib.kda_recurrent_replay(ctypes.byref(_rp()), None) == 9


def _bwd(**kw):
    base = dict(T=128, N=1, H=2, dk=128, dv=128, dtype=kda.KDA_BF16, q=FAKE, k=FAKE + 1024, z=FAKE + 2048,
                v=FAKE + 4096, beta=FAKE + 8192, dt_bias=None, A_log=None, g_min=-5.0, scale=1.0, cu_seqlens=None,
                initial_state=None, grad_o=FAKE + 12288, grad_final_state=None, grad_q=FAKE + 16384,
                grad_k=FAKE + 20480, grad_z=FAKE + 24576, grad_v=FAKE + 28672, grad_beta=FAKE + 32768,
                grad_dt_bias=None, grad_A_log=None, grad_initial_state=None, chunk_size=64, gate_kind=0)
    base.update(kw)
    return kda.ChunkBwdArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(T=1 << 31), 2),                  # T above INT32_MAX
    (dict(dk=96, dv=96), 2),
    (dict(chunk_size=16), 2),
    (dict(dtype=9), 3),
    (dict(N=0), 1),
    (dict(T=130, N=4), 1),
    (dict(g_min=0.0), 1),
    (dict(gate_kind=4), 1),
    (dict(grad_o=None), 1),
    (dict(grad_q=None), 1),
    (dict(grad_q=FAKE), 1),                # a gradient aliases an input
    (dict(grad_k=FAKE + 16384), 1),        # two gradients alias
    (dict(grad_v=FAKE + 28680), 4),
    (dict(grad_beta=FAKE + 32769), 4),
    (dict(grad_initial_state=FAKE + 65540), 4),
])
def test_chunk_bwd_rejects(lib, kw, code):
    assert lib.kda_chunk_bwd(ctypes.byref(_bwd(**kw)), FAKE, 1 << 40, None) == code


def test_chunk_bwd_workspace(lib):
    need = lib.kda_chunk_bwd_workspace_size(128, 1, 2, 128, 128, 64)
    assert need > 2 * 2 * 400 * 1024  # two chunks, two heads, ~0.42 MiB each
    assert lib.kda_chunk_bwd_workspace_size(128, 1, 2, 96, 96, 64) == 0
    assert lib.kda_chunk_bwd(ctypes.byref(_bwd()), FAKE, need - 1, None) == 5
    assert lib.kda_chunk_bwd(ctypes.byref(_bwd()), None, need, None) == 5
    assert lib.kda_chunk_bwd(ctypes.byref(_bwd()), FAKE + 16, need, None) == 4


def test_chunk_bwd_minimum_workspace(lib):
    """One long sequence may run in segments: the minimum is the scratch of a 16-chunk segment plus the
    segments' entering states, far below the one-pass size at T = 1M (where the one pass would not fit a
    GPU); batches of several sequences and short sequences need the one-pass size."""
    lib.kda_chunk_bwd_workspace_size_min.argtypes = [ctypes.c_int64, ctypes.c_int64] + [ctypes.c_int32] * 4
    lib.kda_chunk_bwd_workspace_size_min.restype = ctypes.c_size_t
    full = lib.kda_chunk_bwd_workspace_size(1 << 20, 1, 32, 128, 128, 64)
    small = lib.kda_chunk_bwd_workspace_size_min(1 << 20, 1, 32, 128, 128, 64)
    assert full > 200 * (1 << 30) and 0 < small < 4 * (1 << 30)
    assert small >= 1024 * 32 * 128 * 128 * 4  # the entering states of 1024 segments x 32 heads
    for T, N in ((1 << 20, 2), (1024, 1), (128, 1)):
        assert lib.kda_chunk_bwd_workspace_size_min(T, N, 32, 128, 128, 64) == \
            lib.kda_chunk_bwd_workspace_size(T, N, 32, 128, 128, 64)
    assert lib.kda_chunk_bwd_workspace_size_min(4096, 1, 2, 96, 96, 64) == 0


def test_empty_batch_plan(lib):
    """An empty batch (T = 0) takes the fp32 path whatever its dtype and head size: the chunk plan
    and the output pass, which only passes the states through (there are no tiles to map for the
    tensor-core path).  The epilogue, given, has no tokens to run over."""
    for dt, d in ((torch.bfloat16, 128), (torch.float32, 64), (torch.bfloat16, 64)):
        s = kda.chunk_fwd_schedule(0, 3, 32, d, d, dt)
        assert s == {"fused": False, "team": False, "own_chunks": 0, "team_producers": 0, "seg_len": 0,
                     "kernels": 2}, (dt, d)
        assert kda.chunk_fwd_workspace_size(0, 3, 32, d, d, dt) > 0
    a = kda.ChunkArgs(T=0, N=3, H=32, dk=128, dv=128, dtype=kda.KDA_BF16, chunk_size=64, out_gate=16)
    assert lib.kda_chunk_fwd_kernel_count(ctypes.byref(a)) == 2
    # the same sizes with tokens run three kernels on the fp32 path (plan, intra, output pass)
    assert kda.chunk_fwd_schedule(640, 3, 32, 64, 64, torch.float32)["kernels"] == 3


def test_debug_checks_flags(lib):
    assert lib.kda_set_debug_checks(2) == 1  # unknown flag: KDA_ERR_INVALID_ARG
    assert lib.kda_set_debug_checks(-1) == 1
    assert lib.kda_set_debug_checks(1) == 0
    assert lib.kda_set_debug_checks(0) == 0


def test_profile_events_validation_and_last_cuda_error(lib):
    """kda_set_profile_events rejects a negative count, a count above its table and a NULL array
    with a positive count; (NULL, 0) switches timing off.  kda_last_cuda_error is cleared by reading."""
    arr = (ctypes.c_void_p * 1)()
    assert lib.kda_set_profile_events(None, -1) == 1
    assert lib.kda_set_profile_events(None, 1) == 1
    assert lib.kda_set_profile_events(arr, 1 << 20) == 1
    assert lib.kda_set_profile_events(None, 0) == 0
    lib.kda_last_cuda_error.restype = ctypes.c_int32
    lib.kda_last_cuda_error()
    assert lib.kda_last_cuda_error() == 0


def test_schedule_decisions_for_the_workloads(lib):
    """The latency model's choices for the workloads, on 152 SMs (the host query assumes GB300's
    count when no device is present):
    - T = 4096 x H = 32 takes the fused launch, each chain producing its own first 4 chunks;
    - the 1M-token sequence with 32 heads also takes the fused launch;
    - with 2 heads it splits the state pass instead (few chains on many SMs);
    - the varlen batch (32 sequences x 32 heads) takes the separate kernels."""
    from linear_attention_kda_gb300 import synthetic as syn
    bf = torch.bfloat16
    assert kda.chunk_fwd_schedule(4096, 1, 32, 128, 128, bf) == {"fused": True, "team": False, "own_chunks": 4,
                                                                  "team_producers": 0, "seg_len": 0, "kernels": 1}
    assert kda.chunk_fwd_schedule(1 << 20, 1, 32, 128, 128, bf)["fused"]
    s = kda.chunk_fwd_schedule(1 << 20, 1, 2, 128, 128, bf)
    assert not s["fused"] and s["seg_len"] > 0 and s["kernels"] == 5
    lengths = syn.seq_lengths(syn.VARLEN_32, 1)
    s = kda.chunk_fwd_schedule(sum(lengths), 32, 32, 128, 128, bf, syn.cu_seqlens_of(lengths))
    assert s == {"fused": False, "team": False, "own_chunks": 0, "team_producers": 0, "seg_len": 0, "kernels": 3}
    # the fp32 path and the softplus gate never take the tensor-core schedules
    assert kda.chunk_fwd_schedule(4096, 1, 32, 128, 128, torch.float32)["kernels"] == 3
    assert kda.chunk_fwd_schedule(4096, 1, 32, 128, 128, bf, gate="softplus")["kernels"] == 3
