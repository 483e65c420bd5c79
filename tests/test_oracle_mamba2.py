"""Pins for the Mamba-2 oracle: closed forms, brute force, hand-derived trace.

None of these re-type the oracle's formula: each checks it against a result
fixed by the mathematics (cumulative sums, exponential decay, impulse
response, the skip path) or against scalar extended-precision unrolling.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit

from oracle import mamba2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(rng, S, P, N, steps):
    x = rng.standard_normal((steps, S, P))
    z = rng.standard_normal((steps, S, P))
    B = rng.standard_normal((steps, S, N)) / np.sqrt(N)
    C = rng.standard_normal((steps, S, N)) / np.sqrt(N)
    dt = np.log1p(np.exp(rng.normal(-2.0, 0.5, (steps, S))))
    A = -np.exp(rng.uniform(0, 2.5, S))
    D = rng.standard_normal(S)
    h0 = 0.1 * rng.standard_normal((S, P, N))
    return h0, x, z, B, C, dt, A, D


def test_silu_identities():
    z = np.linspace(-30, 30, 601)
    s = mamba2.silu(z)
    # silu(z) - silu(-z) = z (because sigmoid(z) + sigmoid(-z) = 1)
    np.testing.assert_allclose(s - mamba2.silu(-z), z, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s, z * expit(z), rtol=1e-14, atol=1e-300)
    assert mamba2.silu(0.0) == 0.0


def test_group_of_head():
    assert list(mamba2.group_of_head(128, 8)) == [h // 16 for h in range(128)]
    assert list(mamba2.group_of_head(8, 1)) == [0] * 8
    assert list(mamba2.group_of_head(6, 6)) == list(range(6))
    assert list(mamba2.group_of_head(6, 3)) == [0, 0, 1, 1, 2, 2]


def test_golden_scalar_trace():
    with open(os.path.join(GOLDEN, "mamba2_scalar_trace.json")) as f:
        g = json.load(f)
    h = np.array([[[g["h0"]]]])
    for t in range(len(g["x"])):
        x = np.array([[g["x"][t]]])
        z = np.array([[g["z"][t]]])
        h, y = mamba2.conventional_step(h, x, z, np.array([[g["B"]]]), np.array([[g["C"]]]),
                                        np.array([g["dt"]]), np.array([g["A"]]), np.array([g["D"]]))
        assert h[0, 0, 0] == pytest.approx(g["h"][t], abs=1e-15)
        gate = g["z"][t] * expit(g["z"][t])
        assert y[0, 0] == pytest.approx(g["y_pre_gate"][t] * gate, rel=1e-14)


def test_skip_path_exact(rng):
    """h0 = 0 and B = 0: the state stays 0 and y = D x silu(z)."""
    S, P, N, T = 5, 6, 4, 10
    h0, x, z, B, C, dt, A, D = _rand_problem(rng, S, P, N, T)
    h = np.zeros((S, P, N))
    for t in range(T):
        h, y = mamba2.conventional_step(h, x[t], z[t], 0 * B[t], C[t], dt[t], A, D)
        assert np.all(h == 0)
        np.testing.assert_allclose(y, D[:, None] * x[t] * z[t] * expit(z[t]), rtol=1e-14, atol=1e-15)


def test_A_zero_is_cumulative_sum(rng):
    """A = 0 (dA = 1): h_t = h0 + sum_{k<=t} dt_k x_k B_k^T."""
    S, P, N, T = 3, 5, 7, 12
    h0, x, z, B, C, dt, A, D = _rand_problem(rng, S, P, N, T)
    A = np.zeros(S)
    incr = dt[:, :, None, None] * x[:, :, :, None] * B[:, :, None, :]
    closed = h0[None] + np.cumsum(incr, axis=0)
    h = h0
    for t in range(T):
        h, y = mamba2.conventional_step(h, x[t], z[t], B[t], C[t], dt[t], A, D)
        np.testing.assert_allclose(h, closed[t], rtol=1e-12, atol=1e-13)
        yc = (np.einsum("spn,sn->sp", closed[t], C[t]) + D[:, None] * x[t]) * z[t] * expit(z[t])
        np.testing.assert_allclose(y, yc, rtol=1e-12, atol=1e-13)


def test_pure_decay_exponential(rng):
    """x = 0 with constant dt: h_t = exp(A dt t) h0 (sign and count of the decay)."""
    S, P, N, T = 4, 3, 5, 9
    h0, x, z, B, C, dt, A, D = _rand_problem(rng, S, P, N, T)
    dtc = np.full(S, 0.3)
    h = h0
    for t in range(1, T + 1):
        h, y = mamba2.conventional_step(h, 0 * x[0], z[0], B[0], C[0], dtc, A, D)
        np.testing.assert_allclose(h, np.exp(A * 0.3 * t)[:, None, None] * h0, rtol=1e-13)
        r = np.exp(A * 0.3 * t)[:, None] * np.einsum("spn,sn->sp", h0, C[0])
        np.testing.assert_allclose(y, r * z[0] * expit(z[0]), rtol=1e-12, atol=1e-15)


def test_impulse_response():
    """Zero state, one impulse x_1 = e_p, constant B, C, dt: y_t = e^{A dt (t-1)} dt (B.C) silu(z)."""
    P, N = 3, 4
    A, dt, D = -0.7, 0.25, 0.0
    B = np.array([0.5, -1.0, 2.0, 0.25])
    C = np.array([1.0, 0.5, -0.5, 2.0])
    bc = float(B @ C)
    z = np.array([0.3, -0.2, 1.1])
    h = np.zeros((1, P, N))
    for t in range(1, 8):
        x = np.zeros((1, P))
        if t == 1:
            x[0, 1] = 1.0
        h, y = mamba2.conventional_step(h, x, z[None], B[None], C[None], np.array([dt]), np.array([A]), np.array([D]))
        expect = np.zeros(P)
        expect[1] = np.exp(A * dt * (t - 1)) * dt * bc
        np.testing.assert_allclose(y[0], expect * z * expit(z), rtol=1e-13, atol=1e-16)


def _bruteforce_scalar(h0, x, z, B, C, dt, A, D):
    """Explicit scalar loops in extended precision, one (P, N) problem."""
    ld = np.longdouble
    P, N = h0.shape
    h = [[ld(h0[p, n]) for n in range(N)] for p in range(P)]
    ys = []
    for t in range(x.shape[0]):
        dA = np.exp(ld(dt[t]) * ld(A))
        for p in range(P):
            for n in range(N):
                h[p][n] = dA * h[p][n] + ld(dt[t]) * ld(x[t, p]) * ld(B[t, n])
        y = []
        for p in range(P):
            acc = ld(0)
            for n in range(N):
                acc += h[p][n] * ld(C[t, n])
            zz = ld(z[t, p])
            y.append((acc + ld(D) * ld(x[t, p])) * zz / (ld(1) + np.exp(-zz)))
        ys.append(y)
    return np.array(h, dtype=np.float64), np.array(ys, dtype=np.float64)


def test_bruteforce_tiny_state(rng):
    """P=2, N=3 (non-square, so a transposed operand fails), 40 steps."""
    S, P, N, T = 2, 2, 3, 40
    h0, x, z, B, C, dt, A, D = _rand_problem(rng, S, P, N, T)
    for s in range(S):
        hb, yb = _bruteforce_scalar(h0[s], x[:, s], z[:, s], B[:, s], C[:, s], dt[:, s], A[s], D[s])
        h = h0[s][None]
        for t in range(T):
            h, y = mamba2.conventional_step(h, x[t, s][None], z[t, s][None], B[t, s][None], C[t, s][None],
                                            dt[t, s][None], A[s][None], D[s][None])
            np.testing.assert_allclose(y[0], yb[t], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(h[0], hb, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("m", [1, 2, 5, 16, 32])
def test_replay_equals_conventional(rng, m):
    """The unrolled replay formula equals m conventional steps (state and output)."""
    S, P, N = 3, 6, 10
    h0, x, z, B, C, dt, A, D = _rand_problem(rng, S, P, N, m)
    h = h0
    for t in range(m):
        h, y = mamba2.conventional_step(h, x[t], z[t], B[t], C[t], dt[t], A, D)
    xs, Bs, dts = np.moveaxis(x, 0, 1), np.moveaxis(B, 0, 1), np.moveaxis(dt, 0, 1)
    np.testing.assert_allclose(mamba2.replay_state(h0, xs, Bs, dts, A), h, rtol=1e-12, atol=1e-14)
    yr = mamba2.replay_output(h0, xs, Bs, dts, C[m - 1], z[m - 1], A, D)
    np.testing.assert_allclose(yr, y, rtol=1e-11, atol=1e-13)


def test_layer_groups_match_per_head(rng):
    """conventional_step_layer reads group floor(h*G/H): checked head by head."""
    Bt, H, G, P, N = 2, 6, 3, 4, 5
    h0 = rng.standard_normal((Bt, H, P, N))
    x, z = rng.standard_normal((2, Bt, H, P))
    B, C = rng.standard_normal((2, Bt, G, N))
    dt = rng.uniform(0.05, 0.5, (Bt, H))
    A, D = -rng.uniform(0.5, 2, H), rng.standard_normal(H)
    hl, yl = mamba2.conventional_step_layer(h0, x, z, B, C, dt, A, D)
    for b in range(Bt):
        for hh in range(H):
            g = hh // 2
            hs, ys = mamba2.conventional_step(h0[b, hh], x[b, hh], z[b, hh], B[b, g], C[b, g],
                                              dt[b, hh], A[hh], D[hh])
            np.testing.assert_array_equal(hl[b, hh], hs)
            np.testing.assert_array_equal(yl[b, hh], ys)
