"""Pins of the fp64 oracle against what the Kimi K3 report and the mathematics fix.

None of these tests runs the CUDA path.  Each pin is independent of the
oracle's own code: hand-worked fixtures (tests/golden), closed forms, exact
identities of the delta rule, and brute-force equivalences (chunked form,
segment composition) -- chosen so that a dropped term, a wrong sign, a wrong
index or a transposed operand fails at least one of them.  The mutation
tests at the end plant such mistakes into copies of the recurrence and check
that the pins catch them.
"""
import math

import numpy as np
import pytest

from oracle import c_ref, numpy_ref as R
from tests.golden_io import read_recurrence, read_table

G_MIN = -5.0


# ----------------------------------------------------------------------------- gate (Eq. 5)

def test_gate_golden_numpy_and_c():
    rows = read_table("gate_eq5.txt")
    assert len(rows) == 8
    for z, b, a, gmin, g_exp in rows:
        g_np = float(R.gate(np.array([z]), np.array([b]), a, gmin)[0])
        g_c = c_ref.gate1(z, b, a, gmin)
        assert g_np == pytest.approx(g_exp, rel=1e-14, abs=1e-14)
        assert g_c == pytest.approx(g_exp, rel=1e-14, abs=1e-14)


def test_gate_bounds_symmetry_monotone():
    rng = np.random.default_rng(0)
    z = rng.normal(0, 3, size=(4096,))
    g = R.gate(z, 0.0, 0.0, G_MIN)
    # range (g_min, 0) and alpha = e^g > e^{g_min}  (Eq. 5 text: alpha > e^-5)
    assert np.all(g < 0) and np.all(g > G_MIN)
    assert np.all(np.exp(g) > math.exp(G_MIN))
    # Sigmoid(x) + Sigmoid(-x) = 1  =>  g(z) + g(-z) = g_min
    np.testing.assert_allclose(g + R.gate(-z, 0.0, 0.0, G_MIN), G_MIN, rtol=0, atol=1e-13)
    # strictly decreasing in z for any A_log (e^A > 0)
    zs = np.sort(z)
    for a in (-1.0, 0.0, 0.7):
        gs = R.gate(zs, 0.3, a, G_MIN)
        assert np.all(np.diff(gs) <= 0)
    # limits
    assert R.gate(np.array([-800.0]), 0, 0, G_MIN)[0] == 0.0
    assert R.gate(np.array([800.0]), 0, 0, G_MIN)[0] == G_MIN


# ----------------------------------------------------------------------------- unbounded softplus gate

def test_gate_softplus_golden():
    rows = read_table("gate_softplus.txt")
    assert len(rows) == 8
    for z, b, a, g_exp in rows:
        g = float(R.gate_softplus(np.array([z]), np.array([b]), a)[0])
        assert g == pytest.approx(g_exp, rel=1e-14, abs=1e-300)


def test_gate_softplus_identities_and_unbounded():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 4, size=4096)
    for a in (-0.5, 0.0, 0.8):
        g, gm = R.gate_softplus(x, 0.0, a), R.gate_softplus(-x, 0.0, a)
        # Softplus(x) - Softplus(-x) = x  =>  g(x) - g(-x) = -e^A x
        np.testing.assert_allclose(g - gm, -math.exp(a) * x, rtol=0, atol=1e-12)
        assert np.all(g < 0)
        assert np.all(np.diff(R.gate_softplus(np.sort(x), 0.3, a)) <= 0)  # decreasing in z
    # unbounded below: 0 <= Softplus(x) - x = ln(1 + e^-x) <= e^-x, so g ~ -e^A x and no g_min holds
    for xv in (10.0, 100.0, 1e4):
        g = float(R.gate_softplus(np.array([xv]), 0.0, 0.0)[0])
        assert 0.0 <= -g - xv <= math.exp(-xv) * (1 + 1e-12)
    assert float(R.gate_softplus(np.array([1e4]), 0.0, 0.0)[0]) < 1000 * G_MIN


_SP_MUTANTS = {
    "sign_flipped": lambda z, b, a: np.exp(a) * np.logaddexp(0.0, z + b),
    "scale_inside": lambda z, b, a: -np.logaddexp(0.0, np.exp(a) * (z + b)),
    "bias_outside": lambda z, b, a: -np.exp(a) * (np.logaddexp(0.0, z) + b),
    "log_without_one": lambda z, b, a: -np.exp(a) * (z + b),
    "exp_not_softplus": lambda z, b, a: -np.exp(a) * np.exp(z + b),
}


@pytest.mark.parametrize("mutant", sorted(_SP_MUTANTS))
def test_gate_softplus_fixture_catches_planted_mistakes(mutant):
    f = _SP_MUTANTS[mutant]
    failures = sum(not np.isclose(f(z, b, a), g, rtol=1e-12, atol=1e-300)
                   for z, b, a, g in read_table("gate_softplus.txt"))
    assert failures >= 1, "a planted mistake passed every softplus-gate fixture"


def test_recurrence_total_forgetting():
    """A log-decay far below any bound (alpha = e^g underflows to 0, as the unbounded gate allows)
    erases the state: S_t = beta_t k_t v_t^T and o_t = beta_t (k_t . q_t) v_t, with no inf or NaN."""
    rng = np.random.default_rng(21)
    T, dk, dv = 5, 4, 3
    q, k, v = rng.normal(size=(T, dk)), rng.normal(size=(T, dk)), rng.normal(size=(T, dv))
    beta = rng.uniform(0.2, 0.9, size=T)
    g = np.full((T, dk), -2000.0)
    o, S = R.recurrence(q, k, v, g, beta, S0=rng.normal(size=(dk, dv)))
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    np.testing.assert_allclose(S, beta[-1] * np.outer(k[-1], v[-1]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(o, (beta * np.einsum("tc,tc->t", k, q))[:, None] * v, rtol=1e-13, atol=1e-13)


def test_gate_bound_on_workload_distribution():
    """Every gate value of the bf16 workloads' distribution obeys alpha > e^-5 (Eq. 5)."""
    import torch
    from linear_attention_kda_gb300 import synthetic as syn
    w = syn.PREFILL_4K
    d = syn.make_prefill(w, seed=1, T_override=256)
    g = R.gate(d["z"].float().numpy(), d["dt_bias"].numpy()[None], d["A_log"].numpy()[None, :, None])
    assert g.shape == (256, w.H, w.d)
    assert np.all(g > G_MIN) and np.all(g < 0)
    assert torch.is_tensor(d["q"])


# ----------------------------------------------------------------------------- recurrence (Eq. 1)

def _golden_case(name):
    d = read_recurrence(name)
    dk, dv = d["dk"], d["dv"]
    S0 = np.array(d["S0"]).reshape(dk, dv)
    g = np.log(np.array(d["alpha"]))
    k = np.array(d["k"])
    v = np.array(d["v"]).reshape(-1, dv)
    q = np.array(d["q"])
    beta = np.array(d["beta"])
    o = np.array(d["o"]).reshape(-1, dv)
    ST = np.array(d["ST"]).reshape(dk, dv)
    return q, k, v, g, beta, S0, o, ST


def _c_single(q, k, v, g, beta, S0, scale=1.0):
    T, dk = k.shape
    dv = v.shape[1]
    res, _ = c_ref.forward(q[:, None], k[:, None], v[:, None], np.zeros((T, 1, dk)),
                           beta[:, None], np.zeros((1, dk)), np.zeros(1), [0, T],
                           S0=None if S0 is None else S0[None, None], scale=scale,
                           g_direct=g[:, None], nthreads=1)
    return res[(0, 0)]


@pytest.mark.parametrize("name", ["recurrence_dk2_dv1.txt", "recurrence_dk2_dv2.txt"])
def test_recurrence_golden(name):
    q, k, v, g, beta, S0, o_exp, S_exp = _golden_case(name)
    for o, S in (R.recurrence(q, k, v, g, beta, S0),
                 R.chunked(q, k, v, g, beta, S0, C=1),
                 R.chunked(q, k, v, g, beta, S0, C=2)):
        np.testing.assert_allclose(o, o_exp, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(S, S_exp, rtol=1e-14, atol=1e-14)
    # the C coding reads fp32 inputs (3/5, 4/5 round in fp32), so its match is to ~1e-7
    o, S = _c_single(q, k, v, g, beta, S0)
    np.testing.assert_allclose(o, o_exp, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(S, S_exp, rtol=1e-6, atol=1e-6)
    # scale multiplies the output only
    o2, S2 = R.recurrence(q, k, v, g, beta, S0, scale=0.25)
    np.testing.assert_allclose(o2, 0.25 * o_exp, rtol=1e-14)
    np.testing.assert_allclose(S2, S_exp, rtol=1e-14)


def _rand_head(rng, T, dk, dv, unit_k=True):
    q = rng.normal(size=(T, dk))
    k = rng.normal(size=(T, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
        q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.normal(size=(T, dv))
    g = R.gate(rng.normal(0, 2, size=(T, dk)), 0.0, 0.0)
    beta = 1 / (1 + np.exp(-rng.normal(size=T)))
    S0 = rng.normal(0, 0.5, size=(dk, dv))
    # fp32-representable token inputs, so the C coding (fp32 reader) sees the same values
    f = lambda x: x.astype(np.float32).astype(np.float64)  # noqa: E731
    return f(q), f(k), f(v), g, f(beta), S0


def test_identity_state_when_no_decay_no_write():
    """alpha = 1, beta = 0: S_t = S0 and o_t = S0^T q_t; zero output from a zero state."""
    rng = np.random.default_rng(1)
    q, k, v, g, beta, S0 = _rand_head(rng, 37, 8, 5)
    g0 = np.zeros_like(g)
    b0 = np.zeros_like(beta)
    for o, S in (R.recurrence(q, k, v, g0, b0, S0), _c_single(q, k, v, g0, b0, S0)):
        np.testing.assert_array_equal(S, S0)
        np.testing.assert_allclose(o, q @ S0, rtol=1e-13, atol=1e-15)
    o, S = R.recurrence(q, k, v, g0, b0, None)
    assert np.all(o == 0) and np.all(S == 0)


def test_beta_zero_closed_form():
    """beta = 0: S_t = Diag(prod_{i<=t} alpha_i) S0 exactly (pure decay)."""
    rng = np.random.default_rng(2)
    q, k, v, g, beta, S0 = _rand_head(rng, 29, 6, 4)
    b0 = np.zeros_like(beta)
    o, S = R.recurrence(q, k, v, g, b0, S0)
    G = np.cumsum(g, axis=0)
    np.testing.assert_allclose(S, np.exp(G[-1])[:, None] * S0, rtol=1e-12)
    o_exp = np.stack([(np.exp(G[t])[:, None] * S0).T @ q[t] for t in range(len(q))])
    np.testing.assert_allclose(o, o_exp, rtol=1e-12, atol=1e-15)
    oc, Sc = _c_single(q, k, v, g, b0, S0)
    np.testing.assert_allclose(Sc, S, rtol=1e-12)


def test_beta_one_unit_key_reads_back_value():
    """beta = 1 and |k| = 1: (I - k k^T) k = 0, so S_t^T k_t = v_t for any alpha and S."""
    rng = np.random.default_rng(3)
    q, k, v, g, beta, S0 = _rand_head(rng, 50, 16, 7)
    ones = np.ones_like(beta)
    ku = k / np.linalg.norm(k, axis=1, keepdims=True)  # unit to fp64 precision
    o, _ = R.recurrence(ku, ku, v, g, ones, S0)  # q_t = k_t
    np.testing.assert_allclose(o, v, rtol=1e-11, atol=1e-11)
    # the C coding reads k in fp32, where |k| = 1 only to ~1e-7
    oc, _ = _c_single(ku, ku, v, g, ones, S0)
    np.testing.assert_allclose(oc, v, rtol=1e-5, atol=1e-5)


def test_orthonormal_keys_exact_retrieval():
    """alpha = 1, beta = 1, orthonormal k_1..k_n: S_n^T k_i = v_i for every i."""
    rng = np.random.default_rng(4)
    dk, dv, n = 12, 5, 9
    Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    k = Qm[:, :n].T.copy()
    v = rng.normal(size=(n, dv))
    S0 = rng.normal(size=(dk, dv))
    _, S = R.recurrence(np.zeros((n, dk)), k, v, np.zeros((n, dk)), np.ones(n), S0)
    np.testing.assert_allclose(k @ S, v, rtol=1e-12, atol=1e-12)


def test_scalar_case_closed_form():
    """d_k = d_v = 1: s_t = alpha (1 - beta k^2) s_{t-1} + beta k v,  o_t = s_t q_t."""
    rng = np.random.default_rng(5)
    T = 40
    q, k, v = rng.normal(size=(3, T))
    g = -rng.uniform(0, 5, size=T)
    beta = rng.uniform(0, 1, size=T)
    s = 0.7
    o_exp = []
    for t in range(T):
        s = math.exp(g[t]) * (1 - beta[t] * k[t] ** 2) * s + beta[t] * k[t] * v[t]
        o_exp.append(s * q[t])
    o, S = R.recurrence(q[:, None], k[:, None], v[:, None], g[:, None], beta, np.array([[0.7]]))
    np.testing.assert_allclose(o[:, 0], o_exp, rtol=1e-12)
    np.testing.assert_allclose(S[0, 0], s, rtol=1e-12)


def test_value_columns_are_independent():
    """Permuting the value channels permutes the columns of o and S (Eq. 1 acts from the left)."""
    rng = np.random.default_rng(6)
    q, k, v, g, beta, S0 = _rand_head(rng, 33, 8, 6)
    perm = rng.permutation(6)
    o, S = R.recurrence(q, k, v, g, beta, S0)
    op, Sp = R.recurrence(q, k, v[:, perm], g, beta, S0[:, perm])
    np.testing.assert_allclose(op, o[:, perm], rtol=1e-13)
    np.testing.assert_allclose(Sp, S[:, perm], rtol=1e-13)


def test_key_channel_permutation():
    """Permuting key channels of (q, k, g, S0 rows) leaves o unchanged and permutes S rows."""
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = _rand_head(rng, 33, 8, 6)
    perm = rng.permutation(8)
    o, S = R.recurrence(q, k, v, g, beta, S0)
    op, Sp = R.recurrence(q[:, perm], k[:, perm], v, g[:, perm], beta, S0[perm])
    np.testing.assert_allclose(op, o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(Sp, S[perm], rtol=1e-12, atol=1e-14)


def test_linear_in_values_and_state():
    """(V, S0) -> (O, S_T) is linear for fixed q, k, g, beta."""
    rng = np.random.default_rng(8)
    q, k, v1, g, beta, S1 = _rand_head(rng, 21, 5, 3)
    v2 = rng.normal(size=v1.shape)
    S2 = rng.normal(size=S1.shape)
    a, b = 0.3, -1.7
    o1, T1 = R.recurrence(q, k, v1, g, beta, S1)
    o2, T2 = R.recurrence(q, k, v2, g, beta, S2)
    o3, T3 = R.recurrence(q, k, a * v1 + b * v2, g, beta, a * S1 + b * S2)
    np.testing.assert_allclose(o3, a * o1 + b * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(T3, a * T1 + b * T2, rtol=1e-11, atol=1e-12)


def test_explicit_transition_matrix_product():
    """S_T = M_T ... M_1 S0 + sum_t (M_T..M_{t+1}) beta_t k_t v_t^T with dense
    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t) (section 5.1.2 definition of M_t)."""
    rng = np.random.default_rng(9)
    q, k, v, g, beta, S0 = _rand_head(rng, 15, 6, 4, unit_k=False)
    dk = 6
    Ms = [(np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t])) for t in range(15)]
    S = S0.copy()
    for t in range(15):
        S = Ms[t] @ S + beta[t] * np.outer(k[t], v[t])
    _, S_or = R.recurrence(q, k, v, g, beta, S0)
    np.testing.assert_allclose(S_or, S, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- chunked form (Eq. 3-4)

@pytest.mark.parametrize("C", [1, 2, 3, 16, 64])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_chunked_equals_sequential(C, T):
    rng = np.random.default_rng(100 + 7 * C + T)
    q, k, v, g, beta, S0 = _rand_head(rng, T, 16, 8)
    o, S = R.recurrence(q, k, v, g, beta, S0, scale=0.5)
    oc, Sc = R.chunked(q, k, v, g, beta, S0, C=C, scale=0.5)
    scale_o = np.linalg.norm(o)
    assert np.linalg.norm(oc - o) <= 1e-12 * scale_o
    assert np.linalg.norm(Sc - S) <= 1e-12 * np.linalg.norm(S)


def test_chunked_at_gate_floor_64():
    """g at the floor (-5) for a whole 64-token chunk: 1/Gamma = e^{315}, still exact in fp64."""
    rng = np.random.default_rng(11)
    q, k, v, g, beta, S0 = _rand_head(rng, 128, 8, 4)
    g = np.full_like(g, -4.999)
    o, S = R.recurrence(q, k, v, g, beta, S0)
    oc, Sc = R.chunked(q, k, v, g, beta, S0, C=64)
    assert np.linalg.norm(oc - o) <= 1e-10 * np.linalg.norm(o)


def test_chunked_with_slow_decay_and_correlated_keys():
    """The chunked form far from the identity:
    - slow decays, g about -0.05;
    - keys sharing a common direction, so the strictly lower L of a 64-token chunk has a spectral
      norm of several units.
    It still equals the token recurrence; the UT transform's solve is exact algebra, not a series."""
    rng = np.random.default_rng(23)
    T, dk, dv = 200, 32, 16
    base = rng.normal(size=dk)
    k = rng.normal(size=(T, dk)) + 1.5 * base
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.normal(size=(T, dk))
    v = rng.normal(size=(T, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=T)))
    g = -0.05 * rng.uniform(0.5, 1.5, size=(T, dk))
    S0 = rng.normal(0, 0.1, size=(dk, dv))
    G = np.cumsum(g[:64], axis=0)
    L = beta[:64, None] * np.einsum("rc,ic,ric->ri", k[:64], k[:64], np.exp(G[:, None, :] - G[None, :, :]))
    assert np.linalg.norm(np.tril(L, -1), 2) > 2.0  # the stress is real
    o, S = R.recurrence(q, k, v, g, beta, S0)
    oc, Sc = R.chunked(q, k, v, g, beta, S0, C=64)
    assert np.linalg.norm(oc - o) <= 1e-10 * np.linalg.norm(o)
    assert np.linalg.norm(Sc - S) <= 1e-10 * np.linalg.norm(S)


# ----------------------------------------------------------------------------- KCP (Eq. 17)

def test_segment_composition_equals_one_pass():
    """Section 5.1.2, Eq. 17: fold S <- M_j S + S~_j over segments reproduces one pass."""
    rng = np.random.default_rng(12)
    q, k, v, g, beta, S0 = _rand_head(rng, 90, 8, 5)
    _, S_ref = R.recurrence(q, k, v, g, beta, S0)
    S = S0.copy()
    for a, b in ((0, 17), (17, 40), (40, 41), (41, 90)):
        M, St = R.segment_maps(k[a:b], g[a:b], beta[a:b], v[a:b])
        S = M @ S + St
    np.testing.assert_allclose(S, S_ref, rtol=1e-11, atol=1e-12)


def test_split_resume_equals_one_pass():
    """Final state of a prefix, passed as initial state, continues exactly (prefix reuse, section 5.4.1)."""
    rng = np.random.default_rng(13)
    q, k, v, g, beta, S0 = _rand_head(rng, 77, 8, 5)
    o, S = R.recurrence(q, k, v, g, beta, S0)
    o1, S1 = R.recurrence(q[:30], k[:30], v[:30], g[:30], beta[:30], S0)
    o2, S2 = R.recurrence(q[30:], k[30:], v[30:], g[30:], beta[30:], S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S2, S, rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------- C vs NumPy codings

def test_c_oracle_matches_numpy_varlen():
    rng = np.random.default_rng(14)
    H, dk, dv = 3, 8, 6
    lens = [5, 1, 17, 64, 70]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q = rng.normal(size=(T, H, dk)).astype(np.float32)
    k = (rng.normal(size=(T, H, dk)) / 3).astype(np.float32)
    v = rng.normal(size=(T, H, dv)).astype(np.float32)
    z = rng.normal(0, 2, size=(T, H, dk)).astype(np.float32)
    beta = rng.uniform(0, 1, size=(T, H)).astype(np.float32)
    b = rng.uniform(-1, 1, size=(H, dk)).astype(np.float32)
    A = rng.normal(0, 0.3, size=H).astype(np.float32)
    S0 = rng.normal(0, 0.1, size=(len(lens), H, dk, dv))
    o_np, S_np = R.forward(q, k, v, z, beta, b, A, cu, S0=S0, scale=0.9)
    res, info = c_ref.forward(q, k, v, z, beta, b, A, cu, S0=S0, scale=0.9, nthreads=2)
    assert info["threads"] >= 1
    for n in range(len(lens)):
        for h in range(H):
            o_c, S_c = res[(n, h)]
            np.testing.assert_allclose(o_c, o_np[cu[n]:cu[n + 1], h], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(S_c, S_np[n, h], rtol=1e-12, atol=1e-13)


def test_empty_sequences_and_empty_batch():
    """Eq. 1 over zero tokens takes no step.
    - An empty sequence's final state is its initial state, exactly, in both codings.
    - It has no outputs.
    - The sequences around it come out as if the batch held them alone.
    - An empty batch (T = 0) only passes every state through."""
    rng = np.random.default_rng(11)
    H, d = 2, 4
    for lengths in ([0, 5, 0, 0, 3, 0], [0, 0, 0]):
        T = sum(lengths)
        q, k, v, z = (rng.normal(size=(T, H, d)).astype(np.float32) for _ in range(4))
        beta = rng.uniform(0.1, 0.9, size=(T, H)).astype(np.float32)
        b = rng.uniform(-1, 1, size=(H, d)).astype(np.float32)
        a = rng.normal(0, 0.3, size=H).astype(np.float32)
        S0 = rng.normal(size=(len(lengths), H, d, d))
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        o, ST = R.forward(q, k, v, z, beta, b, a, cu, S0=S0)
        res, _ = c_ref.forward(q, k, v, z, beta, b, a, cu, S0=S0)
        assert o.shape == (T, H, d)
        kept = [n for n, L in enumerate(lengths) if L > 0]
        for n, L in enumerate(lengths):
            for h in range(H):
                if L == 0:
                    assert np.array_equal(ST[n, h], S0[n, h]) and np.array_equal(res[(n, h)][1], S0[n, h])
                    assert res[(n, h)][0].shape == (0, d)
        if kept:
            cu2 = np.concatenate([[0], np.cumsum([lengths[n] for n in kept])]).astype(np.int32)
            o2, ST2 = R.forward(q, k, v, z, beta, b, a, cu2, S0=S0[kept])
            assert np.array_equal(o2, o) and np.array_equal(ST2, ST[kept])


# ----------------------------------------------------------------------------- mutation tests

def _mut_decay_after(q, k, v, g, beta, S0):
    S = S0.copy()
    o = []
    for t in range(len(q)):
        S = S + beta[t] * np.outer(k[t], v[t] - S.T @ k[t])
        S = np.exp(g[t])[:, None] * S
        o.append(S.T @ q[t])
    return np.array(o), S


def _mut_transposed_out(q, k, v, g, beta, S0):
    o, S = R.recurrence(q, k, v, g, beta, S0)
    if S.shape[0] != S.shape[1]:
        return o * 0, S
    return np.array([S_ @ q_ for S_, q_ in zip([S] * len(q), q)]), S


def _mut_decay_value_side(q, k, v, g, beta, S0):
    S = S0.copy()
    o = []
    for t in range(len(q)):
        a = np.exp(g[t])
        Sd = S * a[None, : S.shape[1]] if S.shape[1] == S.shape[0] else S * a[0]
        S = Sd + beta[t] * np.outer(k[t], v[t] - Sd.T @ k[t])
        o.append(S.T @ q[t])
    return np.array(o), S


def _mut_output_before_update(q, k, v, g, beta, S0):
    S = S0.copy()
    o = []
    for t in range(len(q)):
        Sd = np.exp(g[t])[:, None] * S
        o.append(Sd.T @ q[t])
        S = Sd + beta[t] * np.outer(k[t], v[t] - Sd.T @ k[t])
    return np.array(o), S


def _mut_no_beta_in_erase(q, k, v, g, beta, S0):
    S = S0.copy()
    o = []
    for t in range(len(q)):
        Sd = np.exp(g[t])[:, None] * S
        S = Sd - np.outer(k[t], Sd.T @ k[t]) + beta[t] * np.outer(k[t], v[t])
        o.append(S.T @ q[t])
    return np.array(o), S


@pytest.mark.parametrize("mutant", [_mut_decay_after, _mut_transposed_out, _mut_decay_value_side,
                                    _mut_output_before_update, _mut_no_beta_in_erase])
def test_pins_catch_planted_mistakes(mutant):
    failures = 0
    for name in ("recurrence_dk2_dv1.txt", "recurrence_dk2_dv2.txt"):
        q, k, v, g, beta, S0, o_exp, S_exp = _golden_case(name)
        o, S = mutant(q, k, v, g, beta, S0)
        if not (np.allclose(o, o_exp, atol=1e-12) and np.allclose(S, S_exp, atol=1e-12)):
            failures += 1
    assert failures >= 1, "a planted mistake passed every golden fixture"


# ----------------------------------------------------------------------------- output epilogue (Eq. 6)

def _output_gate_rows():
    rows = read_table("output_gate_eq6.txt")
    assert len(rows) == 5
    return [(r[0], r[1:5], r[5:9], r[9:13], r[13:17]) for r in rows]


def test_output_gate_golden():
    for eps, o, g, w, y in _output_gate_rows():
        assert np.allclose(R.output_gate(o, g, w, eps), y, rtol=1e-14, atol=1e-15)


def test_output_gate_constant_vector_closed_form():
    """o = c (all channels) with eps = 0: RMSNorm(o) = sign(c), so y = Sigmoid(g) * w * sign(c)."""
    rng = np.random.default_rng(3)
    for c in (-2.5, 0.125, 7.0):
        g, w = rng.normal(size=16), rng.normal(size=16)
        y = R.output_gate(np.full(16, c), g, w, 0.0)
        assert np.allclose(y, np.sign(c) * w / (1.0 + np.exp(-g)), rtol=1e-14, atol=1e-15)


def test_output_gate_scale_invariant_and_per_head():
    """With eps = 0 the result does not depend on the scale of o; the norm of one head uses only
    that head's channels."""
    rng = np.random.default_rng(4)
    o, g, w = rng.normal(size=(5, 3, 8)), rng.normal(size=(5, 3, 8)), rng.normal(size=(3, 8))
    y = R.output_gate(o, g, w, 0.0)
    assert np.allclose(R.output_gate(o * 37.0, g, w, 0.0), y, rtol=1e-13)
    o2 = o.copy()
    o2[:, 1] *= 5.0
    o2[:, 2] += 1.0
    y2 = R.output_gate(o2, g, w, 0.0)
    assert np.array_equal(y2[:, 0], y[:, 0])
    assert np.allclose(y2[:, 1], y[:, 1], rtol=1e-13)


_OG_MUTANTS = {
    "no_square_root": lambda o, g, w, e: np.asarray(o) / (np.mean(np.square(o)) + e) * w / (1 + np.exp(-np.asarray(g))),
    "sum_not_mean": lambda o, g, w, e: np.asarray(o) / np.sqrt(np.sum(np.square(o)) + e) * w / (1 + np.exp(-np.asarray(g))),
    "gate_sign_flipped": lambda o, g, w, e: np.asarray(o) / np.sqrt(np.mean(np.square(o)) + e) * w / (1 + np.exp(np.asarray(g))),
    "eps_outside_root": lambda o, g, w, e: np.asarray(o) / (np.sqrt(np.mean(np.square(o))) + e) * w / (1 + np.exp(-np.asarray(g))),
    "weight_dropped": lambda o, g, w, e: np.asarray(o) / np.sqrt(np.mean(np.square(o)) + e) / (1 + np.exp(-np.asarray(g))),
}


@pytest.mark.parametrize("mutant", sorted(_OG_MUTANTS))
def test_output_gate_fixture_catches_planted_mistakes(mutant):
    f = _OG_MUTANTS[mutant]
    failures = sum(not np.allclose(f(np.array(o), g, np.array(w), eps), y, rtol=1e-12, atol=1e-12)
                   for eps, o, g, w, y in _output_gate_rows())
    assert failures >= 1, "a planted mistake passed every output-gate fixture"


# ----------------------------------------------------------------------------- speculative replay (section 5.4)

def _tokens(rng, T, dk, dv):
    k = rng.normal(size=(T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    return (rng.normal(size=(T, dk)), k, rng.normal(size=(T, dv)), -rng.uniform(0.0, 1.0, size=(T, dk)),
            rng.uniform(0.1, 0.9, size=T))


def test_replay_without_cache_is_the_recurrence():
    rng = np.random.default_rng(11)
    new = _tokens(rng, 5, 4, 3)
    S0 = rng.normal(size=(4, 3))
    o, S = R.replay(_tokens(rng, 0, 4, 3), 0, new, 5, S0)
    o_ref, S_ref = R.recurrence(*new, S0=S0)
    assert np.allclose(o, o_ref, rtol=1e-14, atol=1e-14) and np.allclose(S, S_ref, rtol=1e-14, atol=1e-14)


def test_replay_commit_is_a_prefix_state_and_drafts_leave_it():
    """The committed state equals the recurrence over accepted cached tokens then committed new ones,
    i.e. the state a one-token-at-a-time decoder would hold; outputs of the new tokens do not depend on
    how many are committed; nothing replayed or committed leaves S0 untouched."""
    rng = np.random.default_rng(12)
    cached, new = _tokens(rng, 4, 5, 3), _tokens(rng, 3, 5, 3)
    S0 = rng.normal(size=(5, 3))
    S = S0.copy()
    for t in range(2):  # two accepted cached drafts, one token at a time
        _, S = R.recurrence(*(x[t:t + 1] for x in cached), S0=S)
    o_ref, _ = R.recurrence(*new, S0=S)
    _, S_after_bonus = R.recurrence(*(x[:1] for x in new), S0=S)
    for nc in range(4):
        o, Sc = R.replay(cached, 2, new, nc, S0)
        assert np.allclose(o, o_ref, rtol=1e-13, atol=1e-13)
    o1, S1 = R.replay(cached, 2, new, 1, S0)
    assert np.allclose(S1, S_after_bonus, rtol=1e-13, atol=1e-13)
    _, Sz = R.replay(cached, 0, new, 0, S0)
    assert np.array_equal(Sz, S0)


# ----------------------------------------------------------------------------- gradients (backward pass)

from oracle import autograd_ref as AG  # noqa: E402


def _bw_case(rng, T=5, dk=3, dv=2):
    k = rng.normal(size=(T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    return dict(q=rng.normal(size=(T, dk)), k=k, v=rng.normal(size=(T, dv)), z=rng.normal(0, 1.5, size=(T, dk)),
                beta=rng.uniform(0.1, 0.9, size=T), b=rng.uniform(-1, 1, size=dk), A_log=float(rng.normal(0, 0.3)),
                S0=rng.normal(0, 0.3, size=(dk, dv)), do=rng.normal(size=(T, dv)), dST=rng.normal(size=(dk, dv)))


def _np_loss(c, gate_kind, scale=1.0):
    """sum(o * do) + sum(S_T * dST) through the NumPy oracle (independent of the torch restatement)."""
    if gate_kind == "softplus":
        g = R.gate_softplus(c["z"], c["b"], c["A_log"])
    else:
        g = R.gate(c["z"], c["b"], c["A_log"], G_MIN)
    o, S = R.recurrence(c["q"], c["k"], c["v"], g, c["beta"], S0=c["S0"], scale=scale)
    return float(np.sum(o * c["do"]) + np.sum(S * c["dST"]))


@pytest.mark.parametrize("gate_kind", ["lower_bound", "softplus"])
def test_autograd_forward_restatement_equals_recurrence(gate_kind):
    import torch
    rng = np.random.default_rng(40)
    c = _bw_case(rng, T=9, dk=4, dv=3)
    t = {n: torch.tensor(np.asarray(x, np.float64)) for n, x in c.items()}
    g = AG.gate_torch(t["z"], t["b"], t["A_log"], G_MIN, gate_kind).numpy()
    g_np = R.gate_softplus(c["z"], c["b"], c["A_log"]) if gate_kind == "softplus" else R.gate(c["z"], c["b"], c["A_log"], G_MIN)
    np.testing.assert_allclose(g, g_np, rtol=1e-14, atol=1e-15)
    o, S = AG.recurrence_torch(t["q"], t["k"], t["v"], torch.tensor(g_np), t["beta"], t["S0"], 0.7)
    o_ref, S_ref = R.recurrence(c["q"], c["k"], c["v"], g_np, c["beta"], S0=c["S0"], scale=0.7)
    np.testing.assert_allclose(o.numpy(), o_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S.numpy(), S_ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("gate_kind", ["lower_bound", "softplus"])
def test_gradients_match_central_differences(gate_kind):
    """Every gradient (q, k, v, z, beta, dt_bias, A_log, S0) against central differences of the
    NumPy forward: error O(h^2) ~ 1e-10 relative."""
    rng = np.random.default_rng(41)
    c = _bw_case(rng)
    gr = AG.head_backward(c["q"], c["k"], c["v"], c["z"], c["beta"], c["b"], c["A_log"], c["S0"], c["do"],
                          c["dST"], G_MIN, 1.0, gate_kind)
    h = 1e-5
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("z", "dz"), ("beta", "dbeta"), ("b", "db"),
                        ("A_log", "dA_log"), ("S0", "dS0")):
        x0 = np.array(c[name], dtype=np.float64)
        fd = np.zeros_like(x0)
        for idx in np.ndindex(x0.shape):
            for sgn in (1.0, -1.0):
                x = x0.copy()
                x[idx] += sgn * h
                cc = dict(c)
                cc[name] = x if x.shape else float(x)
                fd[idx] += sgn * _np_loss(cc, gate_kind) / (2 * h)
        np.testing.assert_allclose(gr[gname], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_gradients_beta_zero_closed_form():
    """beta = 0: S_t = Diag(e^{G_t}) S0 with G_t the running sum of g, o_t = scale S_t^T q_t.  Then
    dS0 = scale sum_t Diag(e^{G_t}) q_t do_t^T + Diag(e^{G_T}) dST, dq_t = scale S_t do_t, and k, v do
    not matter (dk = dv = 0)."""
    rng = np.random.default_rng(42)
    c = _bw_case(rng, T=6, dk=4, dv=3)
    c["beta"] = np.zeros(6)
    sc = 0.5
    gr = AG.head_backward(c["q"], c["k"], c["v"], c["z"], c["beta"], c["b"], c["A_log"], c["S0"], c["do"],
                          c["dST"], G_MIN, sc)
    g = R.gate(c["z"], c["b"], c["A_log"], G_MIN)
    G = np.cumsum(g, axis=0)
    dS0 = sum(sc * np.exp(G[t])[:, None] * np.outer(c["q"][t], c["do"][t]) for t in range(6))
    dS0 = dS0 + np.exp(G[-1])[:, None] * c["dST"]
    np.testing.assert_allclose(gr["dS0"], dS0, rtol=1e-13, atol=1e-14)
    for t in range(6):
        np.testing.assert_allclose(gr["dq"][t], sc * (np.exp(G[t])[:, None] * c["S0"]) @ c["do"][t], rtol=1e-13, atol=1e-14)
    assert np.all(gr["dk"] == 0) and np.all(gr["dv"] == 0)


@pytest.mark.parametrize("gate_kind", ["lower_bound", "softplus"])
def test_packed_gradients_sum_gate_parameters_over_sequences(gate_kind):
    """The packed driver ``backward`` (several sequences, several heads): dt_bias and A_log are shared
    by every sequence of a head, so their gradients are sums over sequences; every other gradient
    belongs to one (token, head) or one (sequence, head).  All of them against central differences
    of the packed NumPy forward (``numpy_ref.forward``, an independent code path), on a batch with an
    empty sequence, so that a per-sequence (rather than summed) or per-head-mixed packing fails."""
    rng = np.random.default_rng(43)
    lengths, H, dk, dv = [3, 0, 4, 2], 2, 3, 2
    T, N = sum(lengths), len(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    k = rng.normal(size=(T, H, dk))
    k /= np.linalg.norm(k, axis=2, keepdims=True)
    c = dict(q=rng.normal(size=(T, H, dk)), k=k, v=rng.normal(size=(T, H, dv)), z=rng.normal(0, 1.5, size=(T, H, dk)),
             beta=rng.uniform(0.1, 0.9, size=(T, H)), dt_bias=rng.uniform(-1, 1, size=(H, dk)),
             A_log=rng.normal(0, 0.3, size=H), S0=rng.normal(0, 0.3, size=(N, H, dk, dv)))
    do, dST = rng.normal(size=(T, H, dv)), rng.normal(size=(N, H, dk, dv))

    def loss(cc):
        o, S = R.forward(cc["q"], cc["k"], cc["v"], cc["z"], cc["beta"], cc["dt_bias"], cc["A_log"], cu, S0=cc["S0"],
                         g_min=G_MIN, scale=0.8, gate_kind=gate_kind)
        return float(np.sum(o * do) + np.sum(S * dST))

    gr = AG.backward(c["q"], c["k"], c["v"], c["z"], c["beta"], c["dt_bias"], c["A_log"], cu, do, S0=c["S0"],
                     dST=dST, g_min=G_MIN, scale=0.8, gate_kind=gate_kind)
    h = 1e-5
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("z", "dz"), ("beta", "dbeta"),
                        ("dt_bias", "ddt_bias"), ("A_log", "dA_log"), ("S0", "dS0")):
        x0 = np.array(c[name], dtype=np.float64)
        fd = np.zeros_like(x0)
        for idx in np.ndindex(x0.shape):
            for sgn in (1.0, -1.0):
                cc = dict(c)
                cc[name] = x0.copy()
                cc[name][idx] += sgn * h
                fd[idx] += sgn * loss(cc) / (2 * h)
        np.testing.assert_allclose(gr[gname], fd, rtol=1e-6, atol=1e-8, err_msg=name)
    # the shared parameters really are sums: each differs from every single sequence's share
    per_seq = [AG.head_backward(c["q"][a:b, 0], c["k"][a:b, 0], c["v"][a:b, 0], c["z"][a:b, 0], c["beta"][a:b, 0],
                                c["dt_bias"][0], c["A_log"][0], c["S0"][n, 0], do[a:b, 0], dST[n, 0], G_MIN, 0.8,
                                gate_kind)["dA_log"] for n, (a, b) in enumerate(zip(cu[:-1], cu[1:]))]
    assert gr["dA_log"][0] == pytest.approx(sum(per_seq), rel=1e-12)
    assert all(abs(gr["dA_log"][0] - s) > 1e-6 for s in per_seq if s != 0)
