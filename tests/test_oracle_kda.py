"""Pins for the Kimi Delta Attention oracle: a hand-derived trace, closed forms
that fix the side and order of the channel-wise decay, the reduction to Gated
DeltaNet, brute force, and the replay formulas against the recurrence."""
import json
import os

import numpy as np
import pytest

from oracle import gdn, kda

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, S, dk, dv, T):
    q = rng.standard_normal((T, S, dk))
    k = rng.standard_normal((T, S, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, S, dv))
    g = -0.3 * np.log1p(np.exp(rng.standard_normal((T, S, dk))))  # per-channel log decay <= 0
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, S))))
    S0 = 0.1 * rng.standard_normal((S, dv, dk))
    return S0, q, k, v, g, beta


def test_golden_1x2_trace():
    with open(os.path.join(GOLDEN, "kda_1x2_trace.json")) as f:
        g = json.load(f)
    S = np.array(g["S0"])[None]
    for t in range(2):
        S, o = kda.conventional_step(S, np.array(g["q"][t])[None], np.array(g["k"][t])[None],
                                     np.array(g["v"][t])[None], np.array(g["g"][t])[None], np.array([g["beta"][t]]))
        np.testing.assert_allclose(S[0], np.array(g["S"][t]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(o[0], np.array(g["o"][t]), rtol=0, atol=1e-15)


def test_beta_zero_decays_each_key_column(rng):
    """beta = 0: S_t = S0 Diag(exp(sum g)): column c of S (key channel c) decays by
    its own factor; dv != dk, so decaying the value side cannot pass."""
    S0, q, k, v, g, beta = _rand(rng, 3, 6, 5, 8)
    S = S0
    for t in range(8):
        S, o = kda.conventional_step(S, q[t], k[t], v[t], g[t], 0 * beta[t])
        gam = np.exp(g[: t + 1].sum(axis=0))  # [S, dk]
        np.testing.assert_allclose(S, S0 * gam[:, None, :], rtol=1e-13)
        np.testing.assert_allclose(o, np.einsum("sij,sj->si", S0, gam * q[t]), rtol=1e-12, atol=1e-16)


def test_delta_rule_write_after_decay(rng):
    """beta = 1, unit k: after the step S k = v exactly, for any decay vector
    (the delta step acts on the decayed state)."""
    S0, q, k, v, g, beta = _rand(rng, 4, 7, 3, 1)
    S, _ = kda.conventional_step(S0, q[0], k[0], v[0], g[0], np.ones(4))
    np.testing.assert_allclose(np.einsum("sij,sj->si", S, k[0]), v[0], rtol=1e-13, atol=1e-14)


def test_erase_keeps_decayed_orthogonal_part(rng):
    """beta = 1, v = 0, unit k: S k = 0, and S q = S0 (alpha * q) for q orthogonal to k."""
    S0, q, k, v, g, beta = _rand(rng, 4, 7, 3, 1)
    kk = k[0]
    qo = q[0] - np.einsum("sj,sj->s", q[0], kk)[:, None] * kk
    S, _ = kda.conventional_step(S0, qo, kk, 0 * v[0], g[0], np.ones(4))
    np.testing.assert_allclose(np.einsum("sij,sj->si", S, kk), 0, atol=1e-14)
    np.testing.assert_allclose(np.einsum("sij,sj->si", S, qo),
                               np.einsum("sij,sj->si", S0, np.exp(g[0]) * qo), rtol=1e-12, atol=1e-15)


def test_uniform_decay_is_gated_deltanet(rng):
    """Equal g over the channels: KDA reduces to the Gated DeltaNet oracle (pinned on its own)."""
    S0, q, k, v, g, beta = _rand(rng, 3, 6, 5, 12)
    gs = g[..., 0]
    Sk, Sg = S0, S0
    for t in range(12):
        Sk, ok = kda.conventional_step(Sk, q[t], k[t], v[t], np.repeat(gs[t][:, None], 6, axis=1), beta[t])
        Sg, og = gdn.conventional_step(Sg, q[t], k[t], v[t], gs[t], beta[t])
        np.testing.assert_allclose(ok, og, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(Sk, Sg, rtol=1e-12, atol=1e-15)


def _bruteforce(S0, q, k, v, g, beta):
    """Scalar extended-precision loops over one (dv, dk) problem: decay each
    column, take the delta step on the decayed state, write."""
    ld = np.longdouble
    dv, dk = S0.shape
    S = [[ld(S0[i, j]) for j in range(dk)] for i in range(dv)]
    outs = []
    for t in range(q.shape[0]):
        bt = ld(beta[t])
        D = [[S[i][j] * np.exp(ld(g[t, j])) for j in range(dk)] for i in range(dv)]
        Dk = [sum((D[i][j] * ld(k[t, j]) for j in range(dk)), ld(0)) for i in range(dv)]
        S = [[D[i][j] + bt * (ld(v[t, i]) - Dk[i]) * ld(k[t, j]) for j in range(dk)] for i in range(dv)]
        outs.append([sum((S[i][j] * ld(q[t, j]) for j in range(dk)), ld(0)) for i in range(dv)])
    return np.array(S, dtype=np.float64), np.array(outs, dtype=np.float64)


def test_bruteforce_tiny(rng):
    """dk=3, dv=2 (non-square), 40 steps, extended precision."""
    S0, q, k, v, g, beta = _rand(rng, 2, 3, 2, 40)
    for s in range(2):
        Sb, ob = _bruteforce(S0[s], q[:, s], k[:, s], v[:, s], g[:, s], beta[:, s])
        S = S0[s][None]
        for t in range(40):
            S, o = kda.conventional_step(S, q[t, s][None], k[t, s][None], v[t, s][None], g[t, s][None],
                                         beta[t, s][None])
            np.testing.assert_allclose(o[0], ob[t], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S[0], Sb, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("m", [1, 2, 7, 16, 32])
def test_replay_equals_conventional(rng, m):
    S0, q, k, v, g, beta = _rand(rng, 3, 9, 6, m)
    S = S0
    Ss = []
    for t in range(m):
        Sp = S
        S, o = kda.conventional_step(S, q[t], k[t], v[t], g[t], beta[t])
        Ss.append(Sp)
    ks, vs = np.moveaxis(k, 0, 1), np.moveaxis(v, 0, 1)
    gs, bs = np.moveaxis(g, 0, 1), np.moveaxis(beta, 0, 1)
    np.testing.assert_allclose(kda.replay_state(S0, ks, vs, gs, bs), S, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(kda.replay_output(S0, ks, vs, gs, bs, q[m - 1]), o, rtol=1e-11, atol=1e-13)
    # each correction is e_t = beta_t (v_t - S_{t-1} (alpha_t * k_t)), from the recurrence's own states
    e = kda.replay_corrections(S0, ks, vs, gs, bs)
    for t in range(m):
        want = beta[t][:, None] * (v[t] - np.einsum("sij,sj->si", Ss[t], np.exp(g[t]) * k[t]))
        np.testing.assert_allclose(e[:, t], want, rtol=1e-11, atol=1e-13)


def test_strong_decay_stays_finite(rng):
    """Decays down to exp(-30) per token over 32 records: the replay forms use
    only differences G_t - G_i with t >= i (no exp of a positive sum)."""
    S0, q, k, v, g, beta = _rand(rng, 2, 8, 4, 32)
    g = -30.0 * rng.random(g.shape)
    S = S0
    for t in range(32):
        S, o = kda.conventional_step(S, q[t], k[t], v[t], g[t], beta[t])
    ks, vs = np.moveaxis(k, 0, 1), np.moveaxis(v, 0, 1)
    gs, bs = np.moveaxis(g, 0, 1), np.moveaxis(beta, 0, 1)
    Sr = kda.replay_state(S0, ks, vs, gs, bs)
    assert np.isfinite(Sr).all()
    np.testing.assert_allclose(Sr, S, rtol=1e-10, atol=1e-13)
