"""Plant plausible mistakes in the oracle (CPU only) and check the pins catch them.

Each mutant replaces one oracle function with a subtly wrong version (a
flipped sign, a dropped term, a transposed operand, an off-by-one step); the
pin tests of that module are then run against it and at least one must fail.
"""
import inspect

import numpy as np
import pytest

import oracle.gdn as gdn
import oracle.mamba2 as mamba2
import test_oracle_gdn as pins_gdn
import test_oracle_mamba2 as pins_m2


def _run_pins(module):
    """Run every test_* function of a pin module; return the names that failed."""
    failed = []
    for name, fn in inspect.getmembers(module, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        cases = [{}]
        if "m" in params:
            cases = [{"m": m} for m in (1, 5, 16)]
        for kw in cases:
            if "rng" in params:
                kw = dict(kw, rng=np.random.default_rng(99))
            try:
                fn(**kw)
            except (AssertionError, ValueError, IndexError):
                failed.append(name)
                break
    return failed


def _m2(variant):
    def step(h, x, z, Bh, Ch, dt, A, D):
        h = np.asarray(h, np.float64)
        dt = np.asarray(dt, np.float64)
        dA = np.exp(-dt * A) if variant == "decay_sign" else np.exp(dt * A)
        inp = (x if variant == "no_dt" else dt[..., None] * x)[..., :, None] * Bh[..., None, :]
        if variant == "decay_on_input":
            h_new = dA[..., None, None] * (h + inp)
        else:
            h_new = dA[..., None, None] * h + inp
        src = h if variant == "output_from_old" else h_new
        Dt = 0.0 if variant == "no_D" else np.asarray(D, np.float64)[..., None]
        gate = 1 / (1 + np.exp(-z)) if variant == "sigmoid_gate" else mamba2.silu(z)
        y = (np.einsum("...pn,...n->...p", src, Ch) + Dt * x) * gate
        if variant == "transpose":
            y = (np.einsum("...pn,...p->...n", h_new, Ch[..., : h_new.shape[-2]]) + Dt * x) * gate
        return h_new, y
    return step


def _gdn(variant):
    def step(S, q, k, v, g, beta):
        S = np.asarray(S, np.float64)
        alpha = np.exp((-1 if variant == "alpha_sign" else 1) * np.asarray(g, np.float64))[..., None, None]
        beta = np.asarray(beta, np.float64)[..., None, None]
        Sk = np.einsum("...ij,...j->...i", S, k)
        erase = beta * Sk[..., :, None] * k[..., None, :]
        write = (1.0 if variant == "no_beta_on_v" else beta) * v[..., :, None] * k[..., None, :]
        if variant == "erase_not_decayed":
            S_new = alpha * S - erase + write
        else:
            S_new = alpha * (S - erase) + write
        o = np.einsum("...ij,...j->...i", S if variant == "output_from_old" else S_new, q)
        if variant == "transpose":
            o = np.einsum("...ij,...i->...j", S_new, q[..., : S_new.shape[-2]])
        return S_new, o
    return step


@pytest.mark.parametrize("variant", ["decay_sign", "no_dt", "decay_on_input", "output_from_old",
                                     "no_D", "sigmoid_gate", "transpose"])
def test_mamba2_pins_catch(monkeypatch, variant):
    monkeypatch.setattr(mamba2, "conventional_step", _m2(variant))
    assert _run_pins(pins_m2), f"mutant {variant} passed every Mamba-2 pin"


@pytest.mark.parametrize("variant", ["alpha_sign", "no_beta_on_v", "erase_not_decayed",
                                     "output_from_old", "transpose"])
def test_gdn_pins_catch(monkeypatch, variant):
    monkeypatch.setattr(gdn, "conventional_step", _gdn(variant))
    assert _run_pins(pins_gdn), f"mutant {variant} passed every GDN pin"


def _wrong_weights(dts, A):
    # off by one: includes a_k itself in the decay of record k
    dts = np.asarray(dts, np.float64)
    a = dts * np.asarray(A, np.float64)[..., None]
    m = dts.shape[-1]
    tail = np.zeros_like(a)
    for k in range(m - 1, -1, -1):
        tail[..., k] = (tail[..., k + 1] if k + 1 < m else 0) + a[..., k]
    return np.exp(a.sum(axis=-1)), dts * np.exp(tail)


def test_replay_weight_mutant_caught(monkeypatch):
    monkeypatch.setattr(mamba2, "replay_weights", _wrong_weights)
    with pytest.raises(AssertionError):
        pins_m2.test_replay_equals_conventional(np.random.default_rng(3), 5)
