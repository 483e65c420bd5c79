"""Pins for the Gated DeltaNet oracle: delta-rule identities, decay closed form,
brute force and a hand-derived trace."""
import json
import os

import numpy as np
import pytest

from oracle import gdn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, S, dk, dv, T):
    q = rng.standard_normal((T, S, dk))
    k = rng.standard_normal((T, S, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, S, dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, S))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, S))))
    S0 = 0.1 * rng.standard_normal((S, dv, dk))
    return S0, q, k, v, g, beta


def test_golden_2x2_trace():
    with open(os.path.join(GOLDEN, "gdn_2x2_trace.json")) as f:
        g = json.load(f)
    S = np.array(g["S0"])[None]
    for t in range(2):
        S, o = gdn.conventional_step(S, np.array(g["q"][t])[None], np.array(g["k"][t])[None],
                                     np.array(g["v"][t])[None], np.array([g["g"][t]]), np.array([g["beta"][t]]))
        np.testing.assert_allclose(S[0], np.array(g["S"][t]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(o[0], np.array(g["o"][t]), rtol=0, atol=1e-15)


def test_beta_zero_alpha_one_constant(rng):
    S0, q, k, v, g, beta = _rand(rng, 3, 6, 5, 8)
    S = S0
    for t in range(8):
        S, o = gdn.conventional_step(S, q[t], k[t], v[t], 0 * g[t], 0 * beta[t])
        np.testing.assert_array_equal(S, S0)
        np.testing.assert_allclose(o, np.einsum("sij,sj->si", S0, q[t]), rtol=1e-14)


def test_beta_zero_pure_decay(rng):
    """beta = 0: S_t = prod(alpha) S0 (checks exp(g), not exp(-g), and the step count)."""
    S0, q, k, v, g, beta = _rand(rng, 3, 6, 5, 8)
    S = S0
    for t in range(8):
        S, o = gdn.conventional_step(S, q[t], k[t], v[t], g[t], 0 * beta[t])
        gam = np.exp(g[: t + 1].sum(axis=0))
        np.testing.assert_allclose(S, gam[:, None, None] * S0, rtol=1e-13)
        np.testing.assert_allclose(o, gam[:, None] * np.einsum("sij,sj->si", S0, q[t]), rtol=1e-12, atol=1e-16)


def test_delta_rule_write(rng):
    """beta = 1, unit k: after the step S k = v exactly, for any alpha."""
    S0, q, k, v, g, beta = _rand(rng, 4, 7, 3, 1)
    S, _ = gdn.conventional_step(S0, q[0], k[0], v[0], g[0], np.ones(4))
    np.testing.assert_allclose(np.einsum("sij,sj->si", S, k[0]), v[0], rtol=1e-13, atol=1e-14)


def test_delta_rule_erase_keeps_orthogonal(rng):
    """beta = 1, v = 0, unit k: S k = 0 and S q = alpha S0 q for q orthogonal to k."""
    S0, q, k, v, g, beta = _rand(rng, 4, 7, 3, 1)
    kk = k[0]
    qo = q[0] - np.einsum("sj,sj->s", q[0], kk)[:, None] * kk
    S, _ = gdn.conventional_step(S0, qo, kk, 0 * v[0], g[0], np.ones(4))
    np.testing.assert_allclose(np.einsum("sij,sj->si", S, kk), 0, atol=1e-14)
    np.testing.assert_allclose(np.einsum("sij,sj->si", S, qo),
                               np.exp(g[0])[:, None] * np.einsum("sij,sj->si", S0, qo), rtol=1e-12, atol=1e-15)


def test_orthonormal_keys_store_values(rng):
    """alpha = 1, beta = 1, orthonormal k_1..k_t: S_t k_i = v_i for i <= t and
    S_t q = S0 q for q orthogonal to every k_i."""
    dk, dv, T = 8, 5, 6
    Q, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Q.T[:T]
    S0 = rng.standard_normal((1, dv, dk))
    vals = rng.standard_normal((T, dv))
    qperp = Q.T[T]
    S = S0
    for t in range(T):
        S, _ = gdn.conventional_step(S, qperp[None], keys[t][None], vals[t][None], np.zeros(1), np.ones(1))
        for i in range(t + 1):
            np.testing.assert_allclose(S[0] @ keys[i], vals[i], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(S[0] @ qperp, S0[0] @ qperp, rtol=1e-12, atol=1e-12)


def _bruteforce(S0, q, k, v, g, beta):
    """Scalar extended-precision loops over one (dv, dk) problem."""
    ld = np.longdouble
    dv, dk = S0.shape
    S = [[ld(S0[i, j]) for j in range(dk)] for i in range(dv)]
    outs = []
    for t in range(q.shape[0]):
        a = np.exp(ld(g[t]))
        bt = ld(beta[t])
        Sk = [sum((S[i][j] * ld(k[t, j]) for j in range(dk)), ld(0)) for i in range(dv)]
        S = [[a * (S[i][j] - bt * Sk[i] * ld(k[t, j])) + bt * ld(v[t, i]) * ld(k[t, j]) for j in range(dk)]
             for i in range(dv)]
        outs.append([sum((S[i][j] * ld(q[t, j]) for j in range(dk)), ld(0)) for i in range(dv)])
    return np.array(S, dtype=np.float64), np.array(outs, dtype=np.float64)


def test_bruteforce_tiny(rng):
    """dk=2, dv=3 (non-square), 40 steps, extended precision."""
    S0, q, k, v, g, beta = _rand(rng, 2, 2, 3, 40)
    for s in range(2):
        Sb, ob = _bruteforce(S0[s], q[:, s], k[:, s], v[:, s], g[:, s], beta[:, s])
        S = S0[s][None]
        for t in range(40):
            S, o = gdn.conventional_step(S, q[t, s][None], k[t, s][None], v[t, s][None], g[t, s][None], beta[t, s][None])
            np.testing.assert_allclose(o[0], ob[t], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S[0], Sb, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("m", [1, 2, 7, 16, 32])
def test_replay_equals_conventional(rng, m):
    S0, q, k, v, g, beta = _rand(rng, 3, 9, 6, m)
    S = S0
    for t in range(m):
        S, o = gdn.conventional_step(S, q[t], k[t], v[t], g[t], beta[t])
    ks, vs = np.moveaxis(k, 0, 1), np.moveaxis(v, 0, 1)
    gs, bs = np.moveaxis(g, 0, 1), np.moveaxis(beta, 0, 1)
    np.testing.assert_allclose(gdn.replay_state(S0, ks, vs, gs, bs), S, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(gdn.replay_output(S0, ks, vs, gs, bs, q[m - 1]), o, rtol=1e-11, atol=1e-13)
