"""Mamba-2 decode step, conventional and replayed, in fp64 (oracle; test-only).

Conventional step (the published ``selective_state_update`` decode step; the
pages name the Mamba-2 layer and say conventional decoding updates, reads and
stores the state every step -- "ReplaySSM Caches Inputs Instead of State...",
section "Why SSM layers slow down hybrid models"). Per sequence, head h of
group g(h), state h[P, N]:

    dA      = exp(dt * A)
    h[p, n] = dA * h[p, n] + dt * x[p] * B[n]
    y[p]    = (sum_n h[p, n] * C[n] + D * x[p]) * silu(z[p])

Replay (same page, section "How ReplaySSM works": output from checkpoint plus
buffer, flush folds the buffer into the checkpoint). With records 1..m since
the checkpoint h0 and a_j = dt_j * A:

    h_m = exp(sum_{j<=m} a_j) * h0 + sum_k exp(sum_{k<j<=m} a_j) * dt_k * x_k B_k^T
    y_m = (h_m C_m + D x_m) * silu(z_m)

Readings where the pages are silent: dt arrives positive (no bias, softplus or
clamp here); A and D are per-head scalars; z gates the output through silu
with no separate norm; head h reads group floor(h * G / H).

Shapes: ``P`` = headdim, ``N`` = dstate, ``G`` = ngroups. Leading axes are
free batch axes. Everything is fp64 numpy.
"""
import numpy as np


def group_of_head(nheads, ngroups):
    """Group index g(h) = floor(h * G / H) for every head h (Mamba-2 grouped B/C)."""
    return (np.arange(nheads) * ngroups) // nheads


def silu(z):
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def conventional_step(h, x, z, Bh, Ch, dt, A, D):
    """One conventional decode step for independent (sequence, head) problems.

    h [..., P, N]; x, z [..., P]; Bh, Ch [..., N] (the head's group row);
    dt, A, D [...] (broadcastable). Returns (h_new, y) with y [..., P].
    """
    h = np.asarray(h, np.float64)
    dt = np.asarray(dt, np.float64)
    dA = np.exp(dt * A)
    h_new = dA[..., None, None] * h + (dt[..., None] * x)[..., :, None] * Bh[..., None, :]
    y = (np.einsum("...pn,...n->...p", h_new, Ch) + np.asarray(D, np.float64)[..., None] * x) * silu(z)
    return h_new, y


def expand_groups(B, nheads):
    """[..., G, N] group rows -> [..., H, N] per-head rows using group_of_head."""
    G = B.shape[-2]
    return B[..., group_of_head(nheads, G), :]


def conventional_step_layer(h, x, z, B, C, dt, A, D):
    """Full-layer conventional step. h [Bt,H,P,N]; x,z [Bt,H,P]; B,C [Bt,G,N];
    dt [Bt,H]; A,D [H]. Returns (h_new, y [Bt,H,P])."""
    H = h.shape[-3]
    return conventional_step(h, x, z, expand_groups(B, H), expand_groups(C, H), dt, A, D)


def replay_weights(dts, A):
    """Decay weights of the unrolled recurrence for a window of m records.

    dts [..., m] (record 1 first), A [...]. Returns (P_m [...], w [..., m]) with
    P_m = exp(sum_j dt_j A) and w_k = dt_k * exp(sum_{k<j<=m} dt_j A).
    """
    dts = np.asarray(dts, np.float64)
    a = dts * np.asarray(A, np.float64)[..., None]
    m = dts.shape[-1]
    # suffix sums over j > k, written as an explicit loop over the window
    tail = np.zeros_like(a)
    for k in range(m - 2, -1, -1):
        tail[..., k] = tail[..., k + 1] + a[..., k + 1]
    Pm = np.exp(a.sum(axis=-1))
    w = dts * np.exp(tail)
    return Pm, w


def replay_state(h0, xs, Bs, dts, A):
    """Checkpoint after folding m records: h_m = P_m h0 + sum_k w_k x_k B_k^T.

    h0 [..., P, N]; xs [..., m, P]; Bs [..., m, N]; dts [..., m]; A [...].
    """
    Pm, w = replay_weights(dts, A)
    h = Pm[..., None, None] * np.asarray(h0, np.float64)
    m = xs.shape[-2]
    for k in range(m):
        h = h + (w[..., k, None] * xs[..., k, :])[..., :, None] * Bs[..., k, None, :]
    return h


def replay_output(h0, xs, Bs, dts, C_m, z_m, A, D):
    """Output of the m-th record from the checkpoint and the window, no state.

    y_m = (P_m (h0 C_m) + sum_k w_k (B_k . C_m) x_k + D x_m) * silu(z_m),
    where record m (the last of xs/Bs/dts) is the current input.
    """
    Pm, w = replay_weights(dts, A)
    r = np.einsum("...pn,...n->...p", np.asarray(h0, np.float64), C_m)
    y = Pm[..., None] * r
    m = xs.shape[-2]
    for k in range(m):
        c_k = np.einsum("...n,...n->...", Bs[..., k, :], C_m)
        y = y + (w[..., k] * c_k)[..., None] * xs[..., k, :]
    y = y + np.asarray(D, np.float64)[..., None] * xs[..., m - 1, :]
    return y * silu(z_m)
