"""Thin ctypes binding of libkda (include/kda.h).

Argument marshalling only: every step of KDA runs inside libkda's CUDA
kernels.  PyTorch supplies device memory (outputs and the prefill workspace
are allocated here with torch) and the current stream.  If libkda is not
built or cannot be loaded, every call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

KDA_F32, KDA_BF16 = 0, 1
# gate of the log-decay (kda_gate_kind_t): Eq. 5 bounded below by g_min, or the unbounded softplus gate
GATE_KINDS = {"lower_bound": 0, "softplus": 1}
_STATUS = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED_SHAPE",
    3: "KDA_ERR_UNSUPPORTED_DTYPE", 4: "KDA_ERR_MISALIGNED", 5: "KDA_ERR_WORKSPACE",
    6: "KDA_ERR_CUDA", 7: "KDA_ERR_BAD_SEQLENS", 8: "KDA_ERR_BAD_STATE_INDEX",
    9: "KDA_ERR_NO_DEVICE", 10: "KDA_ERR_DEVICE_TIMEOUT", 11: "KDA_ERR_BAD_TOKEN_COUNT",
    12: "KDA_ERR_NUMERIC",
}
EXPORTED = ["kda_gate", "kda_chunk_fwd", "kda_chunk_fwd_workspace_size", "kda_recurrent_step",
            "kda_status_string", "kda_get_device_error", "kda_abi_version",
            "kda_set_profile_events", "kda_chunk_fwd_kernel_count", "kda_chunk_fwd_static_ws",
            "kda_last_cuda_error", "kda_chunk_fwd_schedule", "kda_output_gate", "kda_recurrent_replay",
            "kda_chunk_fwd_workspace_size_gate", "kda_chunk_bwd", "kda_chunk_bwd_workspace_size",
            "kda_selftest_bounded_wait", "kda_set_debug_checks", "kda_set_chunk_schedule",
            "kda_chunk_bwd_workspace_size_min"]
STATIC_WORKSPACE_BYTES = 64 << 20

_vp = ctypes.c_void_p
_i64, _i32, _f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float


class GateArgs(ctypes.Structure):
    _fields_ = [("T", _i64), ("N", _i64), ("H", _i32), ("dk", _i32), ("dtype", ctypes.c_int),
                ("z", _vp), ("dt_bias", _vp), ("A_log", _vp), ("g_min", _f32),
                ("chunk_size", _i32), ("cu_seqlens", _vp), ("out", _vp), ("gate_kind", _i32)]


class ChunkArgs(ctypes.Structure):
    _fields_ = [("T", _i64), ("N", _i64), ("H", _i32), ("dk", _i32), ("dv", _i32),
                ("dtype", ctypes.c_int), ("q", _vp), ("k", _vp), ("z", _vp), ("v", _vp),
                ("beta", _vp), ("dt_bias", _vp), ("A_log", _vp), ("g_min", _f32), ("scale", _f32),
                ("cu_seqlens", _vp), ("cu_seqlens_host", _vp), ("initial_state", _vp),
                ("final_state", _vp), ("o", _vp), ("chunk_size", _i32),
                ("out_gate", _vp), ("out_norm_weight", _vp), ("out_norm_eps", _f32), ("gate_kind", _i32)]


class ReplayArgs(ctypes.Structure):
    _fields_ = [("N", _i64), ("H", _i32), ("dk", _i32), ("dv", _i32), ("dtype", ctypes.c_int), ("R", _i32),
                ("rq", _vp), ("rk", _vp), ("rz", _vp), ("rv", _vp), ("rbeta", _vp), ("n_replay", _vp),
                ("M", _i32), ("q", _vp), ("k", _vp), ("z", _vp), ("v", _vp), ("beta", _vp), ("n_commit", _vp),
                ("dt_bias", _vp), ("A_log", _vp), ("g_min", _f32), ("scale", _f32), ("state", _vp),
                ("state_indices", _vp), ("num_slots", _i64), ("o", _vp), ("gate_kind", _i32)]


class ChunkBwdArgs(ctypes.Structure):
    _fields_ = [("T", _i64), ("N", _i64), ("H", _i32), ("dk", _i32), ("dv", _i32), ("dtype", ctypes.c_int),
                ("q", _vp), ("k", _vp), ("z", _vp), ("v", _vp), ("beta", _vp), ("dt_bias", _vp), ("A_log", _vp),
                ("g_min", _f32), ("scale", _f32), ("cu_seqlens", _vp), ("initial_state", _vp), ("grad_o", _vp),
                ("grad_final_state", _vp), ("grad_q", _vp), ("grad_k", _vp), ("grad_z", _vp), ("grad_v", _vp),
                ("grad_beta", _vp), ("grad_dt_bias", _vp), ("grad_A_log", _vp), ("grad_initial_state", _vp),
                ("chunk_size", _i32), ("gate_kind", _i32)]


class OutputGateArgs(ctypes.Structure):
    _fields_ = [("T", _i64), ("H", _i32), ("dv", _i32), ("dtype", ctypes.c_int), ("o", _vp), ("g", _vp),
                ("norm_weight", _vp), ("eps", _f32), ("y", _vp)]


class StepArgs(ctypes.Structure):
    _fields_ = [("N", _i64), ("H", _i32), ("dk", _i32), ("dv", _i32), ("dtype", ctypes.c_int),
                ("q", _vp), ("k", _vp), ("z", _vp), ("v", _vp), ("beta", _vp),
                ("dt_bias", _vp), ("A_log", _vp), ("g_min", _f32), ("scale", _f32),
                ("state", _vp), ("state_indices", _vp), ("num_slots", _i64), ("o", _vp), ("gate_kind", _i32)]


class KDAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {_STATUS.get(int(code), code)}")


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None):
    """Loads libkda.so (raises if missing: build it with linear_attention_kda_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libkda is not built ({p} missing); run "
                               "`python -m linear_attention_kda_gb300.build`")
        L = ctypes.CDLL(p)
        L.kda_gate.argtypes = [ctypes.POINTER(GateArgs), _vp]
        L.kda_gate.restype = ctypes.c_int
        L.kda_chunk_fwd.argtypes = [ctypes.POINTER(ChunkArgs), _vp, ctypes.c_size_t, _vp]
        L.kda_chunk_fwd.restype = ctypes.c_int
        L.kda_chunk_fwd_workspace_size.argtypes = [_i64, _i64, _i32, _i32, _i32, ctypes.c_int, _i32, _vp]
        L.kda_chunk_fwd_workspace_size.restype = ctypes.c_size_t
        L.kda_chunk_fwd_workspace_size_gate.argtypes = [_i64, _i64, _i32, _i32, _i32, ctypes.c_int, _i32, _vp, _i32]
        L.kda_chunk_fwd_workspace_size_gate.restype = ctypes.c_size_t
        L.kda_chunk_bwd_workspace_size.argtypes = [_i64, _i64, _i32, _i32, _i32, _i32]
        L.kda_chunk_bwd_workspace_size.restype = ctypes.c_size_t
        L.kda_chunk_bwd_workspace_size_min.argtypes = [_i64, _i64, _i32, _i32, _i32, _i32]
        L.kda_chunk_bwd_workspace_size_min.restype = ctypes.c_size_t
        L.kda_chunk_bwd.argtypes = [ctypes.POINTER(ChunkBwdArgs), _vp, ctypes.c_size_t, _vp]
        L.kda_chunk_bwd.restype = ctypes.c_int
        L.kda_selftest_bounded_wait.argtypes = [_vp, _vp]
        L.kda_selftest_bounded_wait.restype = ctypes.c_int
        L.kda_recurrent_step.argtypes = [ctypes.POINTER(StepArgs), _vp]
        L.kda_recurrent_step.restype = ctypes.c_int
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_get_device_error.argtypes = [_vp]
        L.kda_get_device_error.restype = ctypes.c_int
        L.kda_abi_version.restype = ctypes.c_int
        L.kda_set_profile_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), _i32]
        L.kda_set_profile_events.restype = ctypes.c_int
        L.kda_chunk_fwd_kernel_count.argtypes = [ctypes.POINTER(ChunkArgs)]
        L.kda_chunk_fwd_kernel_count.restype = _i32
        L.kda_chunk_fwd_schedule.argtypes = [ctypes.POINTER(ChunkArgs), ctypes.POINTER(_i64)]
        L.kda_chunk_fwd_schedule.restype = ctypes.c_int
        L.kda_chunk_fwd_static_ws.argtypes = [ctypes.POINTER(ChunkArgs), _vp]
        L.kda_chunk_fwd_static_ws.restype = ctypes.c_int
        L.kda_set_debug_checks.argtypes = [_i32]
        L.kda_set_debug_checks.restype = ctypes.c_int
        L.kda_set_chunk_schedule.argtypes = [_i32]
        L.kda_set_chunk_schedule.restype = ctypes.c_int
        L.kda_recurrent_replay.argtypes = [ctypes.POINTER(ReplayArgs), _vp]
        L.kda_recurrent_replay.restype = ctypes.c_int
        L.kda_output_gate.argtypes = [ctypes.POINTER(OutputGateArgs), _vp]
        L.kda_output_gate.restype = ctypes.c_int
        L.kda_last_cuda_error.argtypes = []
        L.kda_last_cuda_error.restype = _i32
        _lib = L
        return L


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _gate_kind(gate: str) -> int:
    if gate not in GATE_KINDS:
        raise ValueError(f"gate must be one of {sorted(GATE_KINDS)}")
    return GATE_KINDS[gate]


def _stream(t: torch.Tensor):
    return torch.cuda.current_stream(t.device).cuda_stream


def _check(code: int, where: str):
    if code != 0:
        if code == 6 and _lib is not None:  # KDA_ERR_CUDA
            where = f"{where} (cudaError_t {int(_lib.kda_last_cuda_error())})"
        raise KDAError(code, where)


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def gate(z: torch.Tensor, dt_bias=None, A_log=None, g_min: float = -5.0, chunk_size: int = 0,
         cu_seqlens: Optional[torch.Tensor] = None, n_seq: int = 1, out=None,
         gate: str = "lower_bound") -> torch.Tensor:
    """kda_gate: g = g_min * sigmoid(exp(A_log) (z + dt_bias)) (Eq. 5), or with gate="softplus"
    g = -exp(A_log) * softplus(z + dt_bias); or its chunk-local cumsum."""
    L = load_library()
    T, H, dk = z.shape
    _contig(z, dt_bias, A_log, cu_seqlens)
    if out is None:
        out = torch.empty((T, H, dk), dtype=torch.float32, device=z.device)
    a = GateArgs(T=T, N=(cu_seqlens.numel() - 1) if cu_seqlens is not None else n_seq, H=H, dk=dk,
                 dtype=_dtype_code(z), z=_ptr(z), dt_bias=_ptr(dt_bias), A_log=_ptr(A_log),
                 g_min=g_min, chunk_size=chunk_size, cu_seqlens=_ptr(cu_seqlens), out=_ptr(out),
                 gate_kind=_gate_kind(gate))
    _check(L.kda_gate(ctypes.byref(a), _stream(z)), "kda_gate")
    return out


# below this g_min the bounded gate's bf16 d = 128 prefill runs on the fp32 path (kda.h)
TC_MIN_G_MIN = -5.5


def chunk_fwd_workspace_size(T, N, H, dk, dv, dtype: torch.dtype, chunk_size=64, cu_seqlens_host=None,
                             gate: str = "lower_bound", g_min: float = -5.0):
    """kda_chunk_fwd_workspace_size_gate for the path the call takes (the fp32 path's size, that of the
    softplus gate, for a bounded gate with g_min below TC_MIN_G_MIN)."""
    L = load_library()
    if gate == "lower_bound" and not g_min >= TC_MIN_G_MIN:
        gate = "softplus"
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    hp = None
    if cu_seqlens_host is not None:
        hp = cu_seqlens_host.data_ptr()
    return int(L.kda_chunk_fwd_workspace_size_gate(T, N, H, dk, dv, code, chunk_size, hp, _gate_kind(gate)))


def chunk_fwd(q, k, v, z, beta, dt_bias=None, A_log=None, *, g_min: float = -5.0, scale: float = 1.0,
              cu_seqlens: Optional[torch.Tensor] = None, cu_seqlens_host: Optional[torch.Tensor] = None,
              n_seq: int = 1, initial_state: Optional[torch.Tensor] = None,
              output_final_state: bool = False, final_state: Optional[torch.Tensor] = None,
              chunk_size: int = 64, workspace: Optional[torch.Tensor] = None,
              out: Optional[torch.Tensor] = None, out_gate: Optional[torch.Tensor] = None,
              out_norm_weight: Optional[torch.Tensor] = None, out_norm_eps: float = 1e-6,
              gate: str = "lower_bound"):
    """kda_chunk_fwd: chunkwise KDA prefill (Eq. 1 evaluated as Eq. 3-4).  Returns (o, final_state).
    gate="softplus" selects the unbounded gate (run on the fp32 CUDA-core path).

    With out_gate ([T, H, dv], the gate pre-activation W_g x), o holds the output epilogue of Eq. 6,
    Sigmoid(out_gate) * RMSNorm(o~) (per-head RMSNorm with weight out_norm_weight [H, dv], eps)."""
    L = load_library()
    T, H, dk = q.shape
    dv = v.shape[2]
    _contig(q, k, v, z, beta, dt_bias, A_log, cu_seqlens, initial_state, out_gate, out_norm_weight)
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else n_seq
    if cu_seqlens_host is not None:
        cu_seqlens_host = cu_seqlens_host.to(dtype=torch.int32, device="cpu").contiguous()
    o = out if out is not None else torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    fs = final_state
    if fs is None and output_final_state:
        fs = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    need = chunk_fwd_workspace_size(T, N, H, dk, dv, q.dtype, chunk_size, cu_seqlens_host, gate, g_min)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    a = ChunkArgs(T=T, N=N, H=H, dk=dk, dv=dv, dtype=_dtype_code(q), q=_ptr(q), k=_ptr(k), z=_ptr(z),
                  v=_ptr(v), beta=_ptr(beta), dt_bias=_ptr(dt_bias), A_log=_ptr(A_log), g_min=g_min,
                  scale=scale, cu_seqlens=_ptr(cu_seqlens),
                  cu_seqlens_host=None if cu_seqlens_host is None else cu_seqlens_host.data_ptr(),
                  initial_state=_ptr(initial_state), final_state=_ptr(fs), o=_ptr(o),
                  chunk_size=chunk_size, out_gate=_ptr(out_gate), out_norm_weight=_ptr(out_norm_weight),
                  out_norm_eps=out_norm_eps, gate_kind=_gate_kind(gate))
    _check(L.kda_chunk_fwd(ctypes.byref(a), _ptr(workspace), workspace.numel(), _stream(q)),
           "kda_chunk_fwd")
    return o, fs


def chunk_bwd(q, k, v, z, beta, dt_bias, A_log, grad_o, *, g_min: float = -5.0, scale: float = 1.0,
              cu_seqlens: Optional[torch.Tensor] = None, n_seq: int = 1,
              initial_state: Optional[torch.Tensor] = None, grad_final_state: Optional[torch.Tensor] = None,
              gate: str = "lower_bound", param_grads: bool = True, state_grad: bool = True,
              workspace: Optional[torch.Tensor] = None) -> dict:
    """kda_chunk_bwd: gradients of the chunked prefill given grad_o (and grad_final_state).

    Returns a dict with q, k, v, z, beta (dtype of q) and, when asked, dt_bias, A_log (fp32) and
    initial_state (fp32 [N, H, dk, dv])."""
    L = load_library()
    T, H, dk = q.shape
    dv = v.shape[2]
    _contig(q, k, v, z, beta, dt_bias, A_log, grad_o, cu_seqlens, initial_state, grad_final_state)
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else n_seq
    g = {n: torch.empty_like(x) for n, x in (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta))}
    if param_grads:
        g["dt_bias"] = torch.zeros((H, dk), dtype=torch.float32, device=q.device)
        g["A_log"] = torch.zeros((H,), dtype=torch.float32, device=q.device)
    if state_grad:
        g["initial_state"] = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    if workspace is None:  # a given workspace is used as it is (a smaller one segments a long sequence)
        need = int(L.kda_chunk_bwd_workspace_size(T, N, H, dk, dv, 64))
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    a = ChunkBwdArgs(T=T, N=N, H=H, dk=dk, dv=dv, dtype=_dtype_code(q), q=_ptr(q), k=_ptr(k), z=_ptr(z), v=_ptr(v),
                     beta=_ptr(beta), dt_bias=_ptr(dt_bias), A_log=_ptr(A_log), g_min=g_min, scale=scale,
                     cu_seqlens=_ptr(cu_seqlens), initial_state=_ptr(initial_state), grad_o=_ptr(grad_o),
                     grad_final_state=_ptr(grad_final_state), grad_q=_ptr(g["q"]), grad_k=_ptr(g["k"]),
                     grad_z=_ptr(g["z"]), grad_v=_ptr(g["v"]), grad_beta=_ptr(g["beta"]),
                     grad_dt_bias=_ptr(g.get("dt_bias")), grad_A_log=_ptr(g.get("A_log")),
                     grad_initial_state=_ptr(g.get("initial_state")), chunk_size=64, gate_kind=_gate_kind(gate))
    _check(L.kda_chunk_bwd(ctypes.byref(a), _ptr(workspace), workspace.numel(), _stream(q)), "kda_chunk_bwd")
    return g


def chunk_bwd_workspace_size(T, N, H, dk=128, dv=128, minimum: bool = False) -> int:
    """kda_chunk_bwd_workspace_size (one pass), or with minimum=True kda_chunk_bwd_workspace_size_min
    (the smallest workspace kda_chunk_bwd accepts: segments of one long sequence)."""
    L = load_library()
    f = L.kda_chunk_bwd_workspace_size_min if minimum else L.kda_chunk_bwd_workspace_size
    return int(f(T, N, H, dk, dv, 64))


def output_gate(o, g, norm_weight=None, eps: float = 1e-6, *, out: Optional[torch.Tensor] = None):
    """kda_output_gate: Sigmoid(g) * RMSNorm(o) per (token, head) (Eq. 6 without projections).
    o, g: [T, H, dv]; norm_weight: [H, dv] fp32 or None; out may be o (in place)."""
    L = load_library()
    T, H, dv = o.shape
    _contig(o, g, norm_weight)
    y = out if out is not None else torch.empty_like(o)
    a = OutputGateArgs(T=T, H=H, dv=dv, dtype=_dtype_code(o), o=_ptr(o), g=_ptr(g),
                       norm_weight=_ptr(norm_weight), eps=eps, y=_ptr(y))
    _check(L.kda_output_gate(ctypes.byref(a), _stream(o)), "kda_output_gate")
    return y


def recurrent_step(q, k, v, z, beta, dt_bias, A_log, state, *, g_min: float = -5.0, scale: float = 1.0,
                   state_indices: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   gate: str = "lower_bound"):
    """kda_recurrent_step: one decode token per sequence; `state` is updated in place.  Returns o."""
    L = load_library()
    N, H, dk = q.shape
    dv = v.shape[2]
    _contig(q, k, v, z, beta, dt_bias, A_log, state, state_indices)
    o = out if out is not None else torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    a = StepArgs(N=N, H=H, dk=dk, dv=dv, dtype=_dtype_code(q), q=_ptr(q), k=_ptr(k), z=_ptr(z),
                 v=_ptr(v), beta=_ptr(beta), dt_bias=_ptr(dt_bias), A_log=_ptr(A_log), g_min=g_min,
                 scale=scale, state=_ptr(state), state_indices=_ptr(state_indices),
                 num_slots=state.shape[0], o=_ptr(o), gate_kind=_gate_kind(gate))
    _check(L.kda_recurrent_step(ctypes.byref(a), _stream(q)), "kda_recurrent_step")
    return o


def recurrent_replay(cached, n_replay, new, n_commit, dt_bias, A_log, state, *, g_min: float = -5.0,
                     scale: float = 1.0, state_indices: Optional[torch.Tensor] = None,
                     out: Optional[torch.Tensor] = None, gate: str = "lower_bound"):
    """kda_recurrent_replay: speculative decoding with replay (section 5.4).

    cached: (q, k, z, v, beta) of the cached draft window, [N, R, H, d] / [N, R, H] (or None: R = 0);
    new: (q, k, z, v, beta) of the new tokens, [N, M, H, d] / [N, M, H]; n_replay, n_commit: int32 [N]
    on the device.  Replays the accepted cached tokens, runs the new ones (outputs returned,
    [N, M, H, dv]) and writes back the state after the first n_commit new tokens, in place."""
    L = load_library()
    q, k, z, v, beta = new
    N, M, H, dk = q.shape
    dv = v.shape[3]
    if cached is None:
        rq = rk = rz = rv = rb = None
        R = 0
    else:
        rq, rk, rz, rv, rb = cached
        R = rq.shape[1]
    _contig(q, k, z, v, beta, rq, rk, rz, rv, rb, n_replay, n_commit, dt_bias, A_log, state, state_indices)
    o = out if out is not None else torch.empty((N, M, H, dv), dtype=q.dtype, device=q.device)
    a = ReplayArgs(N=N, H=H, dk=dk, dv=dv, dtype=_dtype_code(q), R=R, rq=_ptr(rq), rk=_ptr(rk), rz=_ptr(rz),
                   rv=_ptr(rv), rbeta=_ptr(rb), n_replay=_ptr(n_replay), M=M, q=_ptr(q), k=_ptr(k), z=_ptr(z),
                   v=_ptr(v), beta=_ptr(beta), n_commit=_ptr(n_commit), dt_bias=_ptr(dt_bias),
                   A_log=_ptr(A_log), g_min=g_min, scale=scale, state=_ptr(state),
                   state_indices=_ptr(state_indices), num_slots=state.shape[0], o=_ptr(o),
                   gate_kind=_gate_kind(gate))
    _check(L.kda_recurrent_replay(ctypes.byref(a), _stream(q)), "kda_recurrent_replay")
    return o


def selftest_bounded_wait(device=None) -> tuple:
    """kda_selftest_bounded_wait: a wait nothing completes must give up on its own.  Returns
    (device error code read afterwards, seconds waited)."""
    L = load_library()
    t = torch.zeros((1,), dtype=torch.int64, device=device or "cuda")
    _check(L.kda_selftest_bounded_wait(_vp(t.data_ptr()), torch.cuda.current_stream(t.device).cuda_stream),
           "kda_selftest_bounded_wait")
    code = get_device_error(t.device)
    return code, int(t.item()) / 1e9


def get_device_error(device=None) -> int:
    """Waits for the current stream and returns (and clears) the device error code (0 = none)."""
    L = load_library()
    return int(L.kda_get_device_error(torch.cuda.current_stream(device).cuda_stream))


CHECK_FINITE = 1
SCHEDULES = {"auto": 0, "separate": 1, "fused": 2, "team": 3}


def set_chunk_schedule(mode: str) -> None:
    """kda_set_chunk_schedule: "auto" (the library's latency model), or force "separate", "fused" or
    "team" where the problem is eligible for it (process-wide; every schedule computes the same result)."""
    _check(load_library().kda_set_chunk_schedule(SCHEDULES[mode]), "kda_set_chunk_schedule")



def set_debug_checks(flags: int) -> None:
    """kda_set_debug_checks: with CHECK_FINITE, every entry point scans what it wrote and sets
    KDA_ERR_NUMERIC (read with get_device_error) on a NaN or an infinity; 0 turns the checks off."""
    _check(load_library().kda_set_debug_checks(int(flags)), "kda_set_debug_checks")


def status_string(code: int) -> str:
    return load_library().kda_status_string(int(code)).decode()


def set_profile_events(events) -> None:
    """Per-kernel timing: pass torch.cuda.Event objects (already recorded once), or [] to stop."""
    L = load_library()
    if not events:
        _check(L.kda_set_profile_events(None, 0), "kda_set_profile_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[int(e.cuda_event) for e in events])
    _check(L.kda_set_profile_events(arr, len(events)), "kda_set_profile_events")


def chunk_fwd_kernel_count(T=0, N=1, H=1, dk=128, dv=128, dtype=torch.bfloat16, cu_seqlens_host=None,
                           gate: str = "lower_bound", out_gate: bool = False, g_min: float = -5.0) -> int:
    """Kernels kda_chunk_fwd launches for these sizes (the split-sequence state pass adds two; with
    out_gate, a separate epilogue pass adds one where the output pass does not apply it)."""
    cu = None
    if cu_seqlens_host is not None:
        cu = cu_seqlens_host.to(dtype=torch.int32, device="cpu").contiguous()
    a = ChunkArgs(T=T, N=N, H=H, dk=dk, dv=dv, dtype=KDA_BF16 if dtype == torch.bfloat16 else KDA_F32,
                  cu_seqlens_host=None if cu is None else cu.data_ptr(), chunk_size=64,
                  gate_kind=_gate_kind(gate), out_gate=16 if out_gate else None, g_min=g_min)
    return int(load_library().kda_chunk_fwd_kernel_count(ctypes.byref(a)))


def chunk_fwd_schedule(T=0, N=1, H=1, dk=128, dv=128, dtype=torch.bfloat16, cu_seqlens_host=None,
                       gate: str = "lower_bound", g_min: float = -5.0) -> dict:
    """The schedule kda_chunk_fwd picks for these sizes (see kda_chunk_fwd_schedule in kda.h)."""
    cu = None
    if cu_seqlens_host is not None:
        cu = cu_seqlens_host.to(dtype=torch.int32, device="cpu").contiguous()
    a = ChunkArgs(T=T, N=N, H=H, dk=dk, dv=dv, dtype=KDA_BF16 if dtype == torch.bfloat16 else KDA_F32,
                  cu_seqlens_host=None if cu is None else cu.data_ptr(), chunk_size=64,
                  gate_kind=_gate_kind(gate), g_min=g_min)
    out = (_i64 * 4)()
    _check(load_library().kda_chunk_fwd_schedule(ctypes.byref(a), out), "kda_chunk_fwd_schedule")
    return {"fused": out[0] == 1, "team": out[0] == 2, "own_chunks": int(out[1]) if out[0] == 1 else 0,
            "team_producers": int(out[1]) if out[0] == 2 else 0, "seg_len": int(out[2]), "kernels": int(out[3])}


def chunk_fwd_static_ws(q, k, v, z, beta, dt_bias=None, A_log=None, *, g_min: float = -5.0,
                        scale: float = 1.0, cu_seqlens: Optional[torch.Tensor] = None,
                        cu_seqlens_host: Optional[torch.Tensor] = None, n_seq: int = 1,
                        initial_state: Optional[torch.Tensor] = None,
                        final_state: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                        gate: str = "lower_bound"):
    """kda_chunk_fwd_static_ws: prefill using the library's own fixed scratch buffer.

    For callers that must not allocate device scratch: outputs (`out`,
    `final_state`) are caller-provided tensors here (allocated by this helper only
    when omitted); the library uses its internal buffer of STATIC_WORKSPACE_BYTES
    and rejects larger problems (KDA_ERR_WORKSPACE).  Calls on one device share
    that buffer, so they must not overlap in time.
    """
    L = load_library()
    T, H, dk = q.shape
    dv = v.shape[2]
    _contig(q, k, v, z, beta, dt_bias, A_log, cu_seqlens, initial_state)
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else n_seq
    if cu_seqlens_host is not None:
        cu_seqlens_host = cu_seqlens_host.to(dtype=torch.int32, device="cpu").contiguous()
    o = out if out is not None else torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    a = ChunkArgs(T=T, N=N, H=H, dk=dk, dv=dv, dtype=_dtype_code(q), q=_ptr(q), k=_ptr(k), z=_ptr(z),
                  v=_ptr(v), beta=_ptr(beta), dt_bias=_ptr(dt_bias), A_log=_ptr(A_log), g_min=g_min,
                  scale=scale, cu_seqlens=_ptr(cu_seqlens),
                  cu_seqlens_host=None if cu_seqlens_host is None else cu_seqlens_host.data_ptr(),
                  initial_state=_ptr(initial_state), final_state=_ptr(final_state), o=_ptr(o),
                  chunk_size=64, gate_kind=_gate_kind(gate))
    _check(L.kda_chunk_fwd_static_ws(ctypes.byref(a), _stream(q)), "kda_chunk_fwd_static_ws")
    return o, final_state
