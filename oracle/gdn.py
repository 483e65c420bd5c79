"""Gated DeltaNet decode step, conventional and replayed, in fp64 (oracle; test-only).

Conventional step (the published gated delta rule; the pages name Gated
DeltaNet as one of the SSM layers -- "ReplaySSM Caches Inputs Instead of
State...", section "Why SSM layers slow down hybrid models"). Per sequence and
head, state S[dv, dk], alpha = exp(g):

    S <- alpha * S (I - beta k k^T) + beta v k^T
    o  = S q

Readings: no 1/sqrt(dk) scaling of q; q, k, v share the head count.

Replay (section "How ReplaySSM works"). The step rewrites as
S_t = alpha_t S_{t-1} + e_t k_t^T with e_t = beta_t (v_t - alpha_t S_{t-1} k_t).
Unrolling from the checkpoint S0 with gamma_t = prod_{j<=t} alpha_j:

    e_t = beta_t (v_t - gamma_t S0 k_t - sum_{i<t} (gamma_t/gamma_i)(k_i . k_t) e_i)
    S_m = gamma_m S0 + sum_{t<=m} (gamma_m/gamma_t) e_t k_t^T
    o_m = gamma_m S0 q_m + sum_{t<=m} (gamma_m/gamma_t)(k_t . q_m) e_t
"""
import numpy as np


def conventional_step(S, q, k, v, g, beta):
    """One conventional step for independent problems.

    S [..., dv, dk]; q, k [..., dk]; v [..., dv]; g, beta [...].
    Returns (S_new, o [..., dv]).
    """
    S = np.asarray(S, np.float64)
    alpha = np.exp(np.asarray(g, np.float64))[..., None, None]
    beta = np.asarray(beta, np.float64)[..., None, None]
    Sk = np.einsum("...ij,...j->...i", S, k)
    S_new = alpha * (S - beta * Sk[..., :, None] * k[..., None, :]) + beta * v[..., :, None] * k[..., None, :]
    o = np.einsum("...ij,...j->...i", S_new, q)
    return S_new, o


def _window_terms(S0, ks, vs, gs, betas):
    """log-decay prefix sums Gp [..., m] and corrections e [..., m, dv] of a window."""
    S0 = np.asarray(S0, np.float64)
    gs = np.asarray(gs, np.float64)
    m = ks.shape[-2]
    Gp = np.zeros_like(gs)
    acc = np.zeros(gs.shape[:-1])
    for t in range(m):
        acc = acc + gs[..., t]
        Gp[..., t] = acc
    e = np.zeros(vs.shape[:-2] + (m, vs.shape[-1]))
    for t in range(m):
        u_t = np.einsum("...ij,...j->...i", S0, ks[..., t, :])
        rhs = vs[..., t, :] - np.exp(Gp[..., t])[..., None] * u_t
        for i in range(t):
            kk = np.einsum("...j,...j->...", ks[..., i, :], ks[..., t, :])
            rhs = rhs - (np.exp(Gp[..., t] - Gp[..., i]) * kk)[..., None] * e[..., i, :]
        e[..., t, :] = np.asarray(betas, np.float64)[..., t, None] * rhs
    return Gp, e


def replay_state(S0, ks, vs, gs, betas):
    """Checkpoint after folding m records: S_m = gamma_m S0 + sum_t (gamma_m/gamma_t) e_t k_t^T."""
    Gp, e = _window_terms(S0, ks, vs, gs, betas)
    m = ks.shape[-2]
    S = np.exp(Gp[..., m - 1])[..., None, None] * np.asarray(S0, np.float64)
    for t in range(m):
        c = np.exp(Gp[..., m - 1] - Gp[..., t])
        S = S + (c[..., None] * e[..., t, :])[..., :, None] * ks[..., t, None, :]
    return S


def replay_output(S0, ks, vs, gs, betas, q_m):
    """Output of record m from the checkpoint and the window, no state written:
    o_m = gamma_m S0 q_m + sum_t (gamma_m/gamma_t)(k_t . q_m) e_t."""
    Gp, e = _window_terms(S0, ks, vs, gs, betas)
    m = ks.shape[-2]
    o = np.exp(Gp[..., m - 1])[..., None] * np.einsum("...ij,...j->...i", np.asarray(S0, np.float64), q_m)
    for t in range(m):
        kq = np.einsum("...j,...j->...", ks[..., t, :], q_m)
        o = o + (np.exp(Gp[..., m - 1] - Gp[..., t]) * kq)[..., None] * e[..., t, :]
    return o
