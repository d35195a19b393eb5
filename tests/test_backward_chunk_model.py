"""CPU checks of the chunkwise backward that the kernels implement (csrc/kda_chunk_bwd.cu).

A NumPy model of the same chunk-level algorithm -- forward records per chunk of 64 tokens, the
state entering each chunk, the state adjoint Lambda over the chunks in reverse, the value-side
contractions with both solves by T^T = (I + L^T)^{-1}, the key side's pairwise A and L terms per
(row, channel), the reverse cumulative sum of dG and the gate's derivative -- is compared with the
fp64 reverse-mode oracle (oracle/autograd_ref.py, the token recurrence differentiated directly):

* in fp64 the two agree to rounding, which checks the chunkwise gradient formulas themselves;
* with bf16 rounding at the operands the tensor-core kernels round (the value side's S, Lambda,
  W, K~, U, A, dO, V~, dV~, dX_U, dX_W; the two chains' state and record images), the gradients
  stay well inside the bf16 I/O tolerance of the GPU tests (1e-2).

The model is test code only: it shares nothing with the kernels and reads no GPU result.
"""
import numpy as np
import torch

from linear_attention_kda_gb300 import synthetic as syn
from oracle import autograd_ref as AG


def _bf(x, on):
    if not on:
        return x
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _tf32(x):
    """Round to 10 mantissa bits (nearest, ties to even), fp32 exponent range."""
    a = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    a = ((a + 0xFFF + ((a >> 13) & 1)) >> 13) << 13
    return a.astype(np.uint32).view(np.float32).astype(np.float64)


def _key_terms_factorised(dA, dL, Q, K, B, G, fmt):
    """The key side's four sums as products of scaled operand images, with the decays split against
    two half references (p0 = 15 for rows 0..31, p1 = 47 for rows 32..63): every factor is the
    exponential of at most 16 tokens of decay, or at most 1.  fmt: operand rounding, 'bf16' or 'tf32'."""
    C = Q.shape[0]
    rnd = (lambda x: _bf(x, True)) if fmt == "bf16" else _tf32
    low = np.tril(np.ones((C, C)), -1)
    h0 = np.arange(C) < 32
    p0, p1 = 15, 47

    def img(X, p, rows, sign):  # X_i e^{sign (G_p - G_i)} on `rows`, zero elsewhere
        out = np.zeros_like(X)
        out[rows] = X[rows] * np.exp(sign * (G[p] - G[rows]))
        return rnd(out)

    k0, k1 = img(K, p0, h0, 1), img(K, p1, np.ones(C, bool), 1)
    q0, q1 = img(Q, p0, h0, -1), img(Q, p1, ~h0, -1)
    bk0, bk1 = img(B[:, None] * K, p0, h0, -1), img(B[:, None] * K, p1, ~h0, -1)
    dAl, dLl = rnd(dA * low), rnd(dL * low)
    ra, rl, ca, cl = (np.zeros_like(K) for _ in range(4))
    for r in range(C):
        p, kk = (p0, k0) if r < 32 else (p1, k1)
        er = np.exp(G[r] - G[p])
        ra[r], rl[r] = er * (dAl[r] @ kk), er * (dLl[r] @ kk)
        ca[r] = np.exp(G[p1] - G[r]) * (dAl[:, r] @ q1)
        cl[r] = np.exp(G[p1] - G[r]) * (dLl[:, r] @ bk1)
        if r < 32:
            ca[r] += np.exp(G[p0] - G[r]) * (dAl[:, r] @ q0)
            cl[r] += np.exp(G[p0] - G[r]) * (dLl[:, r] @ bk0)
    return ra + np.diag(dA)[:, None] * K, rl, ca + np.diag(dA)[:, None] * Q, cl


def chunk_backward(q, k, v, z, beta, b, A_log, do, dST=None, g_min=-5.0, scale=1.0, C=64, rounded=False,
                   key_fmt=None):
    """Gradients of sum(o * do) + sum(S_T * dST) for one (sequence, head), chunk by chunk (Eq. 3-4 form).
    rounded: bf16 operands at the tensor-core kernels' rounding points; key_fmt: the key side's sums as
    factorised products with 'bf16' or 'tf32' operands (None: the kernels' direct pairwise form)."""
    T, dk = q.shape
    dv = v.shape[1]
    eA = np.exp(A_log)
    g = g_min / (1.0 + np.exp(-eA * (z + b)))  # Eq. 5
    nch = (T + C - 1) // C
    tril, low = np.tril(np.ones((C, C))), np.tril(np.ones((C, C)), -1)
    recs, ckpt = [], []
    S = np.zeros((dk, dv))
    for ci in range(nch):
        t0, ln = ci * C, min(C, T - ci * C)
        Q, K, V, B, Gg = (np.zeros((C, dk)), np.zeros((C, dk)), np.zeros((C, dv)), np.zeros(C), np.zeros((C, dk)))
        Q[:ln], K[:ln], V[:ln], B[:ln], Gg[:ln] = q[t0:t0 + ln], k[t0:t0 + ln], v[t0:t0 + ln], beta[t0:t0 + ln], \
            g[t0:t0 + ln]
        G = np.cumsum(Gg, 0)
        E = np.exp(G[:, None, :] - G[None, :, :])  # E[r, i, c] = e^{G_rc - G_ic}
        A = np.einsum('rc,ic,ric->ri', Q, K, E) * tril
        L = B[:, None] * np.einsum('rc,ic,ric->ri', K, K, E) * low
        Tm = np.linalg.inv(np.eye(C) + L)
        W, U = Tm @ (B[:, None] * K * np.exp(G)), Tm @ (B[:, None] * V)
        R = dict(Q=Q, K=K, V=V, B=B, G=G, E=E, A=A, T=Tm, W=W, U=U, Qh=Q * np.exp(G), Kt=K * np.exp(G[-1] - G),
                 gam=np.exp(G[-1]), t0=t0, ln=ln)
        recs.append(R)
        ckpt.append(S.copy())
        Vt = U - _bf(W, rounded) @ _bf(S, rounded)
        S = R['gam'][:, None] * S + _bf(R['Kt'], rounded).T @ _bf(Vt, rounded)
    Lam = np.zeros((dk, dv)) if dST is None else dST.copy()
    lam = [None] * nch
    for ci in reversed(range(nch)):
        R = recs[ci]
        lam[ci] = Lam.copy()
        dO = np.zeros((C, dv))
        dO[:R['ln']] = do[R['t0']:R['t0'] + R['ln']]
        bf = lambda x: _bf(x, rounded)  # noqa: E731
        dVt = bf(R['Kt']) @ bf(Lam) + scale * bf(R['A']).T @ bf(dO)
        Lam = R['gam'][:, None] * Lam + scale * bf(R['Qh']).T @ bf(dO) - bf(R['W']).T @ bf(dVt)
    out = {n: np.zeros_like(x) for n, x in (('dq', q), ('dk', k), ('dv', v), ('dz', z), ('dbeta', beta))}
    out['dS0'] = Lam
    for ci, R in enumerate(recs):
        t0, ln = R['t0'], R['ln']
        bf = lambda x: _bf(x, rounded)  # noqa: E731
        dO = np.zeros((C, dv))
        dO[:ln] = do[t0:t0 + ln]
        S, Lm = bf(ckpt[ci]), bf(lam[ci])
        dOb = bf(dO)
        # value side
        Vt = R['U'] - bf(R['W']) @ S
        dVt = bf(R['Kt']) @ Lm + bf(scale * R['A']).T @ dOb
        dXU = R['T'].T @ dVt
        Vtb, dVtb, dXUb = bf(Vt), bf(dVt), bf(dXU)
        dQh = scale * dOb @ S.T
        dXW = R['T'].T @ (-dVtb @ S.T)
        dKt = Vtb @ Lm.T
        dA = scale * (dOb @ Vtb.T) * tril
        dL = -(dXUb @ bf(R['U']).T + bf(dXW) @ bf(R['W']).T) * low
        dgam = np.sum(ckpt[ci] * lam[ci], 1)
        # key side
        Q, K, B, G, E = R['Q'], R['K'], R['B'], R['G'], R['E']
        if key_fmt:
            ra, rl, ca, cl = _key_terms_factorised(dA, dL, Q, K, B, G, key_fmt)
        else:
            ra = np.einsum('ri,ic,ric->rc', dA * low, K, E) + np.diag(dA)[:, None] * K
            rl = np.einsum('ri,ic,ric->rc', dL * low, K, E)
            ca = np.einsum('ir,ic,ric->rc', dA * low, Q, 1.0 / E) + np.diag(dA)[:, None] * Q
            cl = np.einsum('ir,i,ic,ric->rc', dL * low, B, K, 1.0 / E)
        eG, eL = np.exp(G), np.exp(G[-1] - G)
        ktil = K * eL
        dG = (dXW * B[:, None] * K * eG + dQh * Q * eG - dKt * ktil + Q * ra - K * ca + B[:, None] * K * rl
              - K * cl)
        run = dgam * R['gam'] + np.sum((dKt * ktil)[:ln], 0)
        dg = run[None, :] + np.cumsum(dG[:ln][::-1], 0)[::-1]
        sg = 1.0 / (1.0 + np.exp(-eA * (z[t0:t0 + ln] + b)))
        out['dq'][t0:t0 + ln] = (dQh * eG + ra)[:ln]
        out['dk'][t0:t0 + ln] = (B[:, None] * dXW * eG + dKt * eL + ca + B[:, None] * rl + cl)[:ln]
        out['dv'][t0:t0 + ln] = (B[:, None] * dXU)[:ln]
        out['dz'][t0:t0 + ln] = dg * g_min * sg * (1.0 - sg) * eA
        out['dbeta'][t0:t0 + ln] = (np.sum(K * (eG * dXW + rl), 1) + np.sum(dXU * R['V'], 1))[:ln]
    return out


def _case(T, D, seed):
    q, k, v, beta, z = syn.make_tokens(T, 1, D, D, "bf16", seed, z_std=1.5)
    b, a = syn.make_head_params(1, D, seed, b_range=1.0, alog_std=0.25)
    gen = torch.Generator().manual_seed(seed + 7)
    do = torch.randn((T, 1, D), generator=gen).to(torch.bfloat16)
    dST = torch.randn((D, D), generator=gen).double().numpy() * 0.1
    f = lambda x: x[:, 0].double().numpy()  # noqa: E731
    return (f(q), f(k), f(v), f(z), f(beta), b[0].double().numpy(), float(a[0]), f(do)), dST


def _rel(x, r):
    return float(np.linalg.norm(x - r) / np.linalg.norm(r))


def test_chunkwise_gradient_formulas_equal_exact_gradients():
    """A ragged last chunk (150 = 2 x 64 + 22), d = 64, a final-state gradient: every gradient to 1e-11."""
    args, dST = _case(150, 64, 71)
    ref = AG.head_backward(*args[:7], None, args[7], dST)
    got = chunk_backward(*args, dST=dST)
    for n in ("dq", "dk", "dv", "dz", "dbeta", "dS0"):
        assert _rel(got[n], ref[n]) <= 1e-11, n


def test_tensor_core_rounding_points_leave_headroom():
    """bf16 operands where the tensor-core backward rounds them (value side and both chains), d = 128:
    every gradient within 5e-3 of the exact one, against the 1e-2 the bf16 GPU tests allow."""
    args, dST = _case(200, 128, 52)
    ref = AG.head_backward(*args[:7], None, args[7], dST)
    got = chunk_backward(*args, dST=dST, rounded=True)
    for n in ("dq", "dk", "dv", "dz", "dbeta", "dS0"):
        e = _rel(got[n], ref[n])
        assert 1e-5 < e <= 5e-3, (n, e)


def test_factorised_key_side_needs_tf32():
    """The key side as factorised products (a tensor-core design): exact in fp64 terms, but dG sums
    seven partly cancelling terms, so its operand precision shows in dz: bf16 operands exceed the
    bf16 tolerance, tf32 operands stay inside it (with the other tensor-core rounding points on)."""
    args, dST = _case(200, 128, 52)
    ref = AG.head_backward(*args[:7], None, args[7], dST)
    e_bf = _rel(chunk_backward(*args, dST=dST, rounded=True, key_fmt="bf16")["dz"], ref["dz"])
    e_tf = _rel(chunk_backward(*args, dST=dST, rounded=True, key_fmt="tf32")["dz"], ref["dz"])
    assert e_bf > 1e-2 and e_tf <= 5e-3, (e_bf, e_tf)
