"""Replay (Kimi K3 report section 5.4) computed a second way: the window of replayed and new tokens as one
chunk of the chunkwise form (Eq. 3-4), the new tokens' outputs from one pass over the committed state,
and the state after the first m = n_replay + n_commit tokens from one rank-m update built from the
chunk's first m rows (the UT transform is lower triangular, so those rows depend on the first m tokens
only).  It must equal ``numpy_ref.replay`` (the token recurrence of Eq. 1 run token by token), which
pins that oracle function from an independent route, for both gates and every count including zero.
"""
import numpy as np
import pytest

from oracle import numpy_ref as R


def _replay_as_chunk(cached, n_replay, new, n_commit, S0, scale=1.0):
    parts = [np.concatenate([np.asarray(cached[i], np.float64)[:n_replay], np.asarray(new[i], np.float64)])
             for i in range(5)]
    q, k, v, g, beta = parts
    n = q.shape[0]
    G = np.cumsum(g, 0)
    E = np.exp(G[:, None, :] - G[None, :, :])  # e^{G_t - G_i}, read for i <= t only
    tril, low = np.tril(np.ones((n, n))), np.tril(np.ones((n, n)), -1)
    L = beta[:, None] * np.einsum('tc,ic,tic->ti', k, k, E) * low
    A = np.einsum('tc,ic,tic->ti', q, k, E) * tril
    T = np.linalg.inv(np.eye(n) + L)
    W = T @ (beta[:, None] * k * np.exp(G))
    U = T @ (beta[:, None] * v)
    Vt = U - W @ S0
    o = scale * ((q * np.exp(G)) @ S0 + A @ Vt)
    m = n_replay + n_commit
    if m == 0:
        return o[n_replay:], np.array(S0, dtype=np.float64)
    Kt = k[:m] * np.exp(G[m - 1] - G[:m])
    return o[n_replay:], np.exp(G[m - 1])[:, None] * S0 + Kt.T @ Vt[:m]


@pytest.mark.parametrize("gate", ["lower_bound", "softplus"])
def test_replay_equals_the_window_as_one_chunk(gate):
    rng = np.random.default_rng(17)
    dk, dv = 32, 16
    for _ in range(30):
        Rn, M = int(rng.integers(0, 5)), int(rng.integers(1, 5))
        nr, nc = int(rng.integers(0, Rn + 1)), int(rng.integers(0, M + 1))

        def toks(n):
            q = rng.normal(size=(n, dk))
            k = rng.normal(size=(n, dk))
            q /= np.linalg.norm(q, axis=1, keepdims=True)
            k /= np.linalg.norm(k, axis=1, keepdims=True)
            z = rng.normal(size=(n, dk)) * 1.5
            b = rng.uniform(-1.0, 1.0, dk)
            g = R.gate_softplus(z, b, 0.3) if gate == "softplus" else R.gate(z, b, 0.3, -5.0)
            return q, k, rng.normal(size=(n, dv)), g, 1.0 / (1.0 + np.exp(-rng.normal(size=n)))

        cached, new = toks(Rn), toks(M)
        S0 = rng.normal(size=(dk, dv)) * 0.1
        o_ref, S_ref = R.replay(cached, nr, new, nc, S0, scale=0.5)
        o, S = _replay_as_chunk(cached, nr, new, nc, S0, scale=0.5)
        assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12 * np.abs(o_ref).max())
        assert np.allclose(S, S_ref, rtol=1e-12, atol=1e-12 * np.abs(S_ref).max())
