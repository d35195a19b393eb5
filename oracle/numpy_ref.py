"""fp64 NumPy oracle for Kimi Delta Attention.  TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
import this module; the CUDA path never does.  Every function follows a
passage of the Kimi K3 technical report (section 2.1.1 unless stated):

* ``gate``        -- Eq. 5, with the per-head bias b of Eq. 2 inside the
                     logit: g = g_min * Sigmoid(exp(A_h) * (z + b)).
* ``gate_softplus`` -- the unbounded gate of the earlier Kimi Linear design that
                     section 2.1.1 contrasts Eq. 5 with: g = -exp(A_h) * Softplus(z + b).
* ``recurrence``  -- Eq. 1 token by token, decay before the delta update,
                     output read from the updated state.
* ``chunked``     -- Eq. 3 and Eq. 4: chunkwise parallel form with the UT
                     transform.  The report defers the UT derivation to the
                     Kimi Linear paper; the algebra used here is derived from
                     Eq. 1 (see the function docstring) and is pinned by the
                     test that it equals ``recurrence``.
* ``segment_maps``-- section 5.1.2, Eq. 17: a segment's cumulative transition
                     M and its zero-start state S~, so that S_out = M S_in + S~.
* ``replay``      -- section 5.4 (KDA decode): speculative decoding with replay,
                     the committed state advanced over accepted cached drafts
                     and committed new tokens, outputs for every new token.
* ``output_gate`` -- Eq. 6 without the projections W_o and W_g: the per-head
                     RMSNorm of the recurrent output, then the output gate
                     Sigmoid(g) with g = W_g x given.

All arithmetic is fp64; inputs are upcast as given.  Layout of one head:
q, k [T, d_k]; v [T, d_v]; g [T, d_k]; beta [T]; state S [d_k, d_v]
(row = key channel).
"""
from __future__ import annotations

import numpy as np


def gate(z, b, A_log, g_min=-5.0):
    """Eq. 5 (bias inside, per Eq. 2): g = g_min * sigmoid(exp(A_log) * (z + b)).

    z: [..., d_k]; b broadcastable to z; A_log broadcastable to z[..., :1].
    Returns fp64 log-decay g in [g_min, 0].
    """
    z = np.asarray(z, dtype=np.float64)
    x = np.exp(np.asarray(A_log, dtype=np.float64)) * (z + np.asarray(b, dtype=np.float64))
    with np.errstate(over="ignore"):  # exp(-x) = inf for x << 0 gives g = -0, the exact limit
        return g_min / (1.0 + np.exp(-x))


def gate_softplus(z, b, A_log):
    """The gate Eq. 5 replaces (section 2.1.1: the earlier design's log-decay is unbounded below):
    g = -exp(A_log) * Softplus(z + b), Softplus(x) = ln(1 + e^x), so g lies in (-inf, 0).  The bias
    sits inside, as in the reading of Eq. 5.  Softplus is evaluated as max(x, 0) + ln(1 + e^{-|x|}),
    which equals ln(1 + e^x) and overflows for no x.

    z: [..., d_k]; b broadcastable to z; A_log broadcastable to z[..., :1].  Returns fp64 g.
    """
    x = np.asarray(z, dtype=np.float64) + np.asarray(b, dtype=np.float64)
    sp = np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))
    return -np.exp(np.asarray(A_log, dtype=np.float64)) * sp


def recurrence(q, k, v, g, beta, S0=None, scale=1.0):
    """Eq. 1, one head, token by token in fp64.

    S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t.  Returns (o [T, d_v], S_T [d_k, d_v]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, dv))
    for t in range(T):
        alpha = np.exp(g[t])
        Sd = alpha[:, None] * S                      # Diag(alpha_t) S_{t-1}
        S = Sd + beta[t] * np.outer(k[t], v[t] - Sd.T @ k[t])
        o[t] = scale * (S.T @ q[t])
    return o, S


def chunked(q, k, v, g, beta, S0=None, C=64, scale=1.0):
    """Eq. 3 and Eq. 4, one head, chunk by chunk in fp64.

    Within a chunk (positions r = 1..c) with entering state S:
      Gamma rows gamma^r = prod_{i<=r} alpha_i                       (Eq. 3)
      L[r, i] = beta_r <gamma^r * k_r, k_i / gamma^i>, i < r   (strictly lower)
      T = (I + L)^{-1};  U = T diag(beta) V;  W = T diag(beta) (Gamma * K)
      V~ = U - W S                                    (pseudo-values, Eq. 4 text)
      A = Tril[(Q * Gamma)(K / Gamma)^T]              (diagonal kept, Eq. 4)
      O = (Gamma * Q) S + A V~                                        (Eq. 4)
      S_next = Diag(gamma^c) S + (K * gamma^c / Gamma)^T V~
    Derivation: writing S_r = Diag(gamma^r)(S + sum_{i<=r} (k_i/gamma^i) e_i^T)
    turns Eq. 1 into (I + L) E = diag(beta) V - diag(beta)(Gamma*K) S for the
    per-token corrections e_r, i.e. E = U - W S = V~; reading o_r = S_r^T q_r
    off the same expression gives Eq. 4.  fp64 holds 1/Gamma up to e^{5 c}
    without overflow for c <= 128.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, dv))
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        c = t1 - t0
        Q, K, V, B = q[t0:t1], k[t0:t1], v[t0:t1], beta[t0:t1]
        Gam = np.exp(np.cumsum(g[t0:t1], axis=0))          # [c, d_k], row r = gamma^r
        KG, KiG, QG = K * Gam, K / Gam, Q * Gam
        L = np.tril(B[:, None] * (KG @ KiG.T), -1)
        Tinv = np.linalg.inv(np.eye(c) + L)
        U = Tinv @ (B[:, None] * V)
        W = Tinv @ (B[:, None] * KG)
        Vt = U - W @ S
        A = np.tril(QG @ KiG.T)
        o[t0:t1] = scale * (QG @ S + A @ Vt)
        Ktil = K * (Gam[-1][None, :] / Gam)
        S = Gam[-1][:, None] * S + Ktil.T @ Vt
    return o, S


def segment_maps(k, g, beta, v):
    """Section 5.1.2, Eq. 17: (M, S~) of one segment.

    M = prod_{r <- 1}^{t} M_r with M_r = (I - beta_r k_r k_r^T) Diag(alpha_r),
    obtained by running the recurrence with v = 0 from S = I (d_k x d_k);
    S~ is the state reached from S = 0.  Then S_out = M S_in + S~.
    """
    k = np.asarray(k, np.float64)
    dk = k.shape[1]
    T = k.shape[0]
    zq = np.zeros((T, dk))
    _, M = recurrence(zq, k, np.zeros((T, dk)), g, beta, S0=np.eye(dk))
    _, St = recurrence(zq, k, v, g, beta, S0=None)
    return M, St


def forward(q, k, v, z, beta, dt_bias, A_log, cu_seqlens, S0=None, g_min=-5.0, scale=1.0,
            heads=None, gate_kind="lower_bound"):
    """Packed multi-sequence, multi-head oracle (small cases).  gate_kind "lower_bound" is Eq. 5
    (``gate``), "softplus" the unbounded gate (``gate_softplus``, g_min unused).

    q, k, z [T, H, d_k]; v [T, H, d_v]; beta [T, H]; dt_bias [H, d_k];
    A_log [H]; cu_seqlens [N + 1]; S0 [N, H, d_k, d_v] or None.
    Returns (o [T, H, d_v], S_T [N, H, d_k, d_v]) in fp64; heads outside
    ``heads`` (if given) are left at zero.
    """
    q = np.asarray(q, np.float64)
    T, H, dk = q.shape
    dv = np.asarray(v).shape[2]
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    N = len(cu) - 1
    o = np.zeros((T, H, dv))
    ST = np.zeros((N, H, dk, dv))
    hs = range(H) if heads is None else heads
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        for h in hs:
            zh, bh, ah = np.asarray(z, np.float64)[a:b, h], np.asarray(dt_bias, np.float64)[h], \
                float(np.asarray(A_log, np.float64)[h])
            g = gate_softplus(zh, bh, ah) if gate_kind == "softplus" else gate(zh, bh, ah, g_min)
            s0 = None if S0 is None else np.asarray(S0, np.float64)[n, h]
            o[a:b, h], ST[n, h] = recurrence(q[a:b, h], np.asarray(k, np.float64)[a:b, h],
                                             np.asarray(v, np.float64)[a:b, h], g,
                                             np.asarray(beta, np.float64)[a:b, h], s0, scale)
    return o, ST


def output_gate(o, g, w=None, eps=1e-6):
    """Eq. 6 (section 2.1.1) without the projections: y = Sigmoid(g) * RMSNorm(o~), where the RMSNorm
    is taken per head (the report: a per-head RMSNorm of the recurrent output),
        RMSNorm(o~)_c = w_c * o~_c / sqrt(mean_{c'} o~_{c'}^2 + eps)
    over the d_v value channels of one (token, head).

    o, g: [..., d_v] (the last axis is one head's value channels); w: RMSNorm weight broadcastable
    to o (ones when None); eps > 0 (the report gives no value: a parameter).  Returns fp64 y.
    """
    o = np.asarray(o, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    normed = o / np.sqrt(ms + eps)
    if w is not None:
        normed = normed * np.asarray(w, dtype=np.float64)
    with np.errstate(over="ignore"):
        return normed / (1.0 + np.exp(-g))


def replay(cached, n_replay, new, n_commit, S0, scale=1.0):
    """Section 5.4 (KDA decode): speculative decoding with replay, one (sequence, head).

    cached, new: tuples (q, k, v, g, beta) of the cached draft window and of the new tokens (bonus
    token, then the next drafts), token-major.  From the committed state S0: the first n_replay cached
    tokens are replayed (Eq. 1), then every new token runs (Eq. 1) and yields an output; the committed
    state is the one reached after the replayed tokens and the first n_commit new tokens (S0 itself when
    there are none).  Returns (o_new [M, d_v], S_committed [d_k, d_v]).
    """
    parts = [np.concatenate([np.asarray(cached[i], np.float64)[:n_replay], np.asarray(new[i], np.float64)])
             for i in range(5)]
    o, _ = recurrence(*parts, S0=S0, scale=scale)
    m = n_replay + n_commit
    if m == 0:
        S = np.array(S0, dtype=np.float64)
    else:
        _, S = recurrence(*(x[:m] for x in parts), S0=S0, scale=scale)
    return o[n_replay:], S
