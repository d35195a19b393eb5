"""fp64 gradients of Kimi Delta Attention.  TEST INFRASTRUCTURE ONLY.

The Kimi K3 technical report describes the forward pass only; its backward pass (section 5.1.1:
the FlashKDA kernels also serve training) is not written out on the pages.  The reference
gradients here are therefore the exact derivatives of the forward definition: the token
recurrence of Eq. 1 (section 2.1.1) and the gate (Eq. 5, or the unbounded softplus gate), restated
in fp64 PyTorch and differentiated by reverse-mode automatic differentiation.  No blocking,
chunking or reordering beyond the definition.  The restatement is pinned against
``numpy_ref.recurrence`` (same forward values) and its gradients against central finite
differences of ``numpy_ref`` (an independent code path) in the CPU tests.

Only the tests and the package smoke check import this module; the CUDA path never does.
"""
from __future__ import annotations

import numpy as np
import torch


def _t(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float64), dtype=torch.float64)


def gate_torch(z, b, A_log, g_min=-5.0, gate_kind="lower_bound"):
    """Eq. 5, g = g_min * Sigmoid(e^A (z + b)); or the softplus gate g = -e^A * Softplus(z + b)."""
    if gate_kind == "softplus":
        return -torch.exp(A_log) * torch.nn.functional.softplus(z + b)
    return g_min * torch.sigmoid(torch.exp(A_log) * (z + b))


def recurrence_torch(q, k, v, g, beta, S0, scale=1.0):
    """Eq. 1 token by token (one head): S' = Diag(e^{g_t}) S, S = S' + beta_t k_t (v_t - S'^T k_t)^T,
    o_t = scale * S^T q_t.  Returns (o [T, d_v], S_T)."""
    S = S0
    outs = []
    for t in range(q.shape[0]):
        Sp = torch.exp(g[t])[:, None] * S
        e = beta[t] * (v[t] - Sp.T @ k[t])
        S = Sp + torch.outer(k[t], e)
        outs.append(scale * (S.T @ q[t]))
    o = torch.stack(outs) if outs else torch.zeros((0, v.shape[1]), dtype=torch.float64)
    return o, S


def head_backward(q, k, v, z, beta, b, A_log, S0, do, dST=None, g_min=-5.0, scale=1.0,
                  gate_kind="lower_bound"):
    """Gradients of  sum(o * do) + sum(S_T * dST)  for one (sequence, head).

    q, k, z [T, d_k]; v [T, d_v]; beta [T]; b [d_k] (dt_bias row); A_log scalar; S0 [d_k, d_v]
    (None = zero); do [T, d_v]; dST [d_k, d_v] or None.  Returns a dict of fp64 arrays:
    dq, dk, dv, dz, dbeta, db (this head's dt_bias row), dA_log (scalar), dS0, and o, S_T.
    """
    dk_, dv_ = np.asarray(q).shape[1], np.asarray(v).shape[1]
    leaves = {n: _t(x).requires_grad_(True) for n, x in
              (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta), ("b", b), ("A_log", A_log),
               ("S0", np.zeros((dk_, dv_)) if S0 is None else S0))}
    g = gate_torch(leaves["z"], leaves["b"], leaves["A_log"], g_min, gate_kind)
    o, ST = recurrence_torch(leaves["q"], leaves["k"], leaves["v"], g, leaves["beta"], leaves["S0"], scale)
    loss = (o * _t(do)).sum()
    if dST is not None:
        loss = loss + (ST * _t(dST)).sum()
    loss.backward()
    out = {"d" + n: (x.grad if x.grad is not None else torch.zeros_like(x)).numpy() for n, x in leaves.items()}
    out["o"], out["S_T"] = o.detach().numpy(), ST.detach().numpy()
    return out


def backward(q, k, v, z, beta, dt_bias, A_log, cu_seqlens, do, S0=None, dST=None, g_min=-5.0, scale=1.0,
             gate_kind="lower_bound", heads=None):
    """Packed multi-sequence, multi-head gradients (small cases), layouts as ``numpy_ref.forward``:
    q, k, z [T, H, d_k]; v [T, H, d_v]; beta [T, H]; dt_bias [H, d_k]; A_log [H]; do [T, H, d_v];
    S0, dST [N, H, d_k, d_v] or None.  Returns dq, dk, dz [T, H, d_k]; dv [T, H, d_v]; dbeta [T, H];
    ddt_bias [H, d_k]; dA_log [H]; dS0 [N, H, d_k, d_v] (fp64; heads outside ``heads`` left zero)."""
    q, k, v, z, beta, do = (np.asarray(x, np.float64) for x in (q, k, v, z, beta, do))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    N = len(cu) - 1
    r = {"dq": np.zeros((T, H, dk)), "dk": np.zeros((T, H, dk)), "dz": np.zeros((T, H, dk)),
         "dv": np.zeros((T, H, dv)), "dbeta": np.zeros((T, H)), "ddt_bias": np.zeros((H, dk)),
         "dA_log": np.zeros(H), "dS0": np.zeros((N, H, dk, dv))}
    bias = np.zeros((H, dk)) if dt_bias is None else np.asarray(dt_bias, np.float64)
    alog = np.zeros(H) if A_log is None else np.asarray(A_log, np.float64)
    for n in range(N):
        a, e = cu[n], cu[n + 1]
        for h in (range(H) if heads is None else heads):
            s0 = None if S0 is None else np.asarray(S0, np.float64)[n, h]
            dst = None if dST is None else np.asarray(dST, np.float64)[n, h]
            g = head_backward(q[a:e, h], k[a:e, h], v[a:e, h], z[a:e, h], beta[a:e, h], bias[h], alog[h],
                              s0, do[a:e, h], dst, g_min, scale, gate_kind)
            r["dq"][a:e, h], r["dk"][a:e, h], r["dv"][a:e, h] = g["dq"], g["dk"], g["dv"]
            r["dz"][a:e, h], r["dbeta"][a:e, h] = g["dz"], g["dbeta"]
            r["ddt_bias"][h] += g["db"]
            r["dA_log"][h] += g["dA_log"]
            r["dS0"][n, h] = g["dS0"]
    return r
