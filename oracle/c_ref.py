"""ctypes wrapper of the plain-C fp64 oracle (kda_oracle.c).  TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
load this library.  The C code follows the Kimi K3 technical report,
section 2.1.1, Eq. 1 (recurrence, decay before the delta update) and Eq. 5
(bounded gate with the bias of Eq. 2 inside the logit).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


class Problem(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64), ("dk", ctypes.c_int64), ("dv", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("z", ctypes.c_void_p),
        ("stride_q", ctypes.c_int64), ("stride_k", ctypes.c_int64),
        ("stride_v", ctypes.c_int64), ("stride_z", ctypes.c_int64),
        ("beta", ctypes.c_void_p), ("stride_beta", ctypes.c_int64),
        ("bias", ctypes.c_void_p),
        ("A_log", ctypes.c_double), ("g_min", ctypes.c_double), ("scale", ctypes.c_double),
        ("S0", ctypes.c_void_p), ("o", ctypes.c_void_p), ("S", ctypes.c_void_p),
        ("g_direct", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into oracle/_build/libkda_oracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC,
                           "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.kda_oracle_run.restype = ctypes.c_int
            L.kda_oracle_run.argtypes = [ctypes.c_int64, ctypes.POINTER(Problem), ctypes.c_int]
            L.kda_oracle_gate1.restype = ctypes.c_double
            L.kda_oracle_gate1.argtypes = [ctypes.c_double] * 4
            L.kda_oracle_problem_size.restype = ctypes.c_int
            assert L.kda_oracle_problem_size() == ctypes.sizeof(Problem), "struct layout mismatch"
            _lib = L
    return _lib


def _f32(x):
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def gate1(z, b, A_log, g_min=-5.0) -> float:
    return lib().kda_oracle_gate1(float(z), float(b), float(A_log), float(g_min))


def forward(q, k, v, z, beta, dt_bias, A_log, cu_seqlens, S0=None, g_min=-5.0, scale=1.0,
            units=None, nthreads=None, g_direct=None):
    """Runs the fp64 oracle on (sequence, head) units of a packed batch.

    q, k, z [T, H, d_k]; v [T, H, d_v]; beta [T, H]; dt_bias [H, d_k]; A_log [H];
    cu_seqlens [N + 1]; S0 [N, H, d_k, d_v] or None.  Tensors may be torch
    (any float dtype; converted exactly to fp32) or numpy.
    ``g_direct`` [T, H, d_k] (fp64) bypasses the gate (for pins on Eq. 1 alone).
    Returns (results, info): results[(n, h)] = (o [len, d_v] fp64, S_T [d_k, d_v] fp64);
    info = {"threads": used, "seconds": wall time of the C call}.
    """
    q, k, v, z, beta = _f32(q), _f32(k), _f32(v), _f32(z), _f32(beta)
    b = _f32(dt_bias)
    a = np.asarray(_f32(A_log), dtype=np.float64)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = [int(x) for x in np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens)]
    N = len(cu) - 1
    s0 = None
    if S0 is not None:
        s0 = S0.detach().cpu().double().numpy() if hasattr(S0, "detach") else np.asarray(S0, np.float64)
        s0 = np.ascontiguousarray(s0)
    gd = None if g_direct is None else np.ascontiguousarray(np.asarray(g_direct, np.float64))
    if units is None:
        units = [(n, h) for n in range(N) for h in range(H)]
    probs = (Problem * len(units))()
    keep = []
    out = {}
    for i, (n, h) in enumerate(units):
        t0, t1 = cu[n], cu[n + 1]
        L = t1 - t0
        o = np.zeros((max(L, 1), dv), np.float64)
        S = np.zeros((dk, dv), np.float64)
        out[(n, h)] = (o[:L], S)
        P = probs[i]
        P.T, P.dk, P.dv = L, dk, dv
        P.q = q.ctypes.data + 4 * (t0 * H * dk + h * dk)
        P.k = k.ctypes.data + 4 * (t0 * H * dk + h * dk)
        P.v = v.ctypes.data + 4 * (t0 * H * dv + h * dv)
        P.z = z.ctypes.data + 4 * (t0 * H * dk + h * dk)
        P.stride_q = P.stride_k = P.stride_z = H * dk
        P.stride_v = H * dv
        P.beta = beta.ctypes.data + 4 * (t0 * H + h)
        P.stride_beta = H
        P.bias = b.ctypes.data + 4 * h * dk
        P.A_log, P.g_min, P.scale = float(a[h]), float(g_min), float(scale)
        P.S0 = None if s0 is None else s0.ctypes.data + 8 * ((n * H + h) * dk * dv)
        P.o = o.ctypes.data
        P.S = S.ctypes.data
        if gd is not None:
            gh = np.ascontiguousarray(gd[t0:t1, h])
            keep.append(gh)
            P.g_direct = gh.ctypes.data
        else:
            P.g_direct = None
        keep.append(o)
    nt = int(nthreads) if nthreads else (os.cpu_count() or 1)
    t_start = time.perf_counter()
    used = lib().kda_oracle_run(len(units), probs, nt)
    secs = time.perf_counter() - t_start
    return out, {"threads": int(used), "seconds": secs}
