"""Kimi Delta Attention (KDA) decode step, conventional and replayed, in fp64
(oracle; test-only).

The pages name KDA as the SSM layer of hybrid models ("ReplaySSM Caches Inputs
Instead of State...", section "Why SSM layers slow down hybrid models") and say
that a serving stack added ReplaySSM to its KDA decode kernel ("ReplaySSM"
repository page, section "Adoption"); they print no equation for it. Reading:
the published KDA recurrence, the gated delta rule whose decay is a vector over
the key channels instead of one scalar per head. Per sequence and head, state
S[dv, dk], alpha = exp(g) with g [dk] (g <= 0):

    S <- S Diag(alpha) (I - beta k k^T) + beta v k^T
    o  = S q

Gated DeltaNet is the case of one g shared by all channels. No 1/sqrt(dk)
scaling of q (as for Gated DeltaNet).

Replay (section "How ReplaySSM works"). The step rewrites as
S_t = S_{t-1} Diag(alpha_t) + e_t k_t^T with
e_t = beta_t (v_t - S_{t-1} (alpha_t * k_t)) (* is the channel-wise product).
Unrolling from the checkpoint S0 with G_t = sum_{j<=t} g_j (a vector over the
channels) and the decayed key k_i^(t) = k_i * exp(G_t - G_i):

    e_t = beta_t (v_t - S0 (exp(G_t) * k_t) - sum_{i<t} (k_i^(t) . k_t) e_i)
    S_m = S0 Diag(exp(G_m)) + sum_{t<=m} e_t (k_t^(m))^T
    o_m = S0 (exp(G_m) * q_m) + sum_{t<=m} (k_t^(m) . q_m) e_t
"""
import numpy as np


def conventional_step(S, q, k, v, g, beta):
    """One conventional step for independent problems.

    S [..., dv, dk]; q, k, g [..., dk]; v [..., dv]; beta [...].
    Returns (S_new, o [..., dv]).
    """
    S = np.asarray(S, np.float64)
    k = np.asarray(k, np.float64)
    alpha = np.exp(np.asarray(g, np.float64))
    beta = np.asarray(beta, np.float64)[..., None, None]
    Sd = S * alpha[..., None, :]                      # S Diag(alpha): column c scaled by alpha[c]
    Sdk = np.einsum("...ij,...j->...i", Sd, k)
    S_new = Sd - beta * Sdk[..., :, None] * k[..., None, :] + beta * np.asarray(v, np.float64)[..., :, None] * k[..., None, :]
    o = np.einsum("...ij,...j->...i", S_new, np.asarray(q, np.float64))
    return S_new, o


def _window_terms(S0, ks, vs, gs, betas):
    """Channel-wise log-decay prefix sums Gp [..., m, dk] and corrections e [..., m, dv]."""
    S0 = np.asarray(S0, np.float64)
    ks = np.asarray(ks, np.float64)
    gs = np.asarray(gs, np.float64)
    m = ks.shape[-2]
    Gp = np.zeros_like(gs)
    acc = np.zeros(gs.shape[:-2] + gs.shape[-1:])
    for t in range(m):
        acc = acc + gs[..., t, :]
        Gp[..., t, :] = acc
    e = np.zeros(vs.shape[:-2] + (m, vs.shape[-1]))
    for t in range(m):
        u_t = np.einsum("...ij,...j->...i", S0, np.exp(Gp[..., t, :]) * ks[..., t, :])
        rhs = np.asarray(vs, np.float64)[..., t, :] - u_t
        for i in range(t):
            kd = ks[..., i, :] * np.exp(Gp[..., t, :] - Gp[..., i, :])
            kk = np.einsum("...j,...j->...", kd, ks[..., t, :])
            rhs = rhs - kk[..., None] * e[..., i, :]
        e[..., t, :] = np.asarray(betas, np.float64)[..., t, None] * rhs
    return Gp, e


def replay_state(S0, ks, vs, gs, betas):
    """Checkpoint after folding m records: S_m = S0 Diag(exp(G_m)) + sum_t e_t (k_t^(m))^T."""
    Gp, e = _window_terms(S0, ks, vs, gs, betas)
    ks = np.asarray(ks, np.float64)
    m = ks.shape[-2]
    S = np.asarray(S0, np.float64) * np.exp(Gp[..., m - 1, :])[..., None, :]
    for t in range(m):
        kd = ks[..., t, :] * np.exp(Gp[..., m - 1, :] - Gp[..., t, :])
        S = S + e[..., t, :, None] * kd[..., None, :]
    return S


def replay_output(S0, ks, vs, gs, betas, q_m):
    """Output of record m from the checkpoint and the window, no state written:
    o_m = S0 (exp(G_m) * q_m) + sum_t (k_t^(m) . q_m) e_t."""
    Gp, e = _window_terms(S0, ks, vs, gs, betas)
    ks = np.asarray(ks, np.float64)
    q_m = np.asarray(q_m, np.float64)
    m = ks.shape[-2]
    o = np.einsum("...ij,...j->...i", np.asarray(S0, np.float64), np.exp(Gp[..., m - 1, :]) * q_m)
    for t in range(m):
        kd = ks[..., t, :] * np.exp(Gp[..., m - 1, :] - Gp[..., t, :])
        o = o + np.einsum("...j,...j->...", kd, q_m)[..., None] * e[..., t, :]
    return o


def replay_corrections(S0, ks, vs, gs, betas):
    """The corrections e_t [..., m, dv] of a window's records (what the ring keeps)."""
    return _window_terms(S0, ks, vs, gs, betas)[1]
