"""Plant plausible mistakes in the oracle (CPU only) and check the pins catch them.

Each mutant replaces one oracle function with a subtly wrong version (a
flipped sign, a dropped term, a transposed operand, an off-by-one step); the
pin tests of that module are then run against it and at least one must fail.
"""
import inspect

import numpy as np
import pytest

import oracle.gdn as gdn
import oracle.kda as kda
import oracle.mamba2 as mamba2
import test_oracle_gdn as pins_gdn
import test_oracle_kda as pins_kda
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
        for mark in getattr(fn, "pytestmark", []):   # a pin's own parametrize cases
            if mark.name == "parametrize":
                names = [n.strip() for n in mark.args[0].split(",")]
                cases = [dict(zip(names, v if len(names) > 1 else (v,))) for v in mark.args[1]]
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


def _kda(variant):
    def step(S, q, k, v, g, beta):
        S = np.asarray(S, np.float64)
        k = np.asarray(k, np.float64)
        g = np.asarray(g, np.float64)
        if variant == "scalar_decay":  # one mean decay per head instead of one per channel
            g = np.repeat(g.mean(axis=-1, keepdims=True), g.shape[-1], axis=-1)
        alpha = np.exp(-g if variant == "alpha_sign" else g)
        beta = np.asarray(beta, np.float64)[..., None, None]
        if variant == "decay_value_side":
            Sd = alpha[..., :, None] * S
        else:
            Sd = S * alpha[..., None, :]
        write = (1.0 if variant == "no_beta_on_v" else beta) * np.asarray(v, np.float64)[..., :, None] * k[..., None, :]
        if variant == "decay_after_delta":
            Sk = np.einsum("...ij,...j->...i", S, k)
            S_new = (S - beta * Sk[..., :, None] * k[..., None, :]) * alpha[..., None, :] + write
        elif variant == "erase_not_decayed":
            Sk = np.einsum("...ij,...j->...i", S, k)
            S_new = Sd - beta * Sk[..., :, None] * k[..., None, :] + write
        else:
            Sdk = np.einsum("...ij,...j->...i", Sd, k)
            S_new = Sd - beta * Sdk[..., :, None] * k[..., None, :] + write
        o = np.einsum("...ij,...j->...i", S if variant == "output_from_old" else S_new, np.asarray(q, np.float64))
        return S_new, o
    return step


@pytest.mark.parametrize("variant", ["alpha_sign", "scalar_decay", "decay_value_side", "decay_after_delta",
                                     "erase_not_decayed", "no_beta_on_v", "output_from_old"])
def test_kda_pins_catch(monkeypatch, variant):
    monkeypatch.setattr(kda, "conventional_step", _kda(variant))
    with np.errstate(over="ignore", invalid="ignore"):  # a growing mutant may overflow on the strong-decay pin
        failed = _run_pins(pins_kda)
    assert failed, f"mutant {variant} passed every KDA pin"


def _kda_undecayed_keys(S0, ks, vs, gs, betas):
    # drops the channel-wise decay of earlier keys in the corrections' coupling terms
    S0 = np.asarray(S0, np.float64)
    ks = np.asarray(ks, np.float64)
    gs = np.asarray(gs, np.float64)
    m = ks.shape[-2]
    Gp = np.cumsum(gs, axis=-2)
    e = np.zeros(vs.shape[:-2] + (m, vs.shape[-1]))
    for t in range(m):
        rhs = vs[..., t, :] - np.einsum("...ij,...j->...i", S0, np.exp(Gp[..., t, :]) * ks[..., t, :])
        for i in range(t):
            rhs = rhs - np.einsum("...j,...j->...", ks[..., i, :], ks[..., t, :])[..., None] * e[..., i, :]
        e[..., t, :] = np.asarray(betas, np.float64)[..., t, None] * rhs
    return Gp, e


def test_kda_replay_mutant_caught(monkeypatch):
    monkeypatch.setattr(kda, "_window_terms", _kda_undecayed_keys)
    with pytest.raises(AssertionError):
        pins_kda.test_replay_equals_conventional(np.random.default_rng(3), 5)


# ----------------------------------------------------------------------------- read-copy rounding

import oracle.readcopy as readcopy  # noqa: E402
import test_oracle_readcopy as pins_rc  # noqa: E402


def _round_mutant(variant):
    real = readcopy.round_rne

    def rnd(x, fmt, saturate=False):
        p, emin, vmax = fmt
        if variant == "half_away":       # ties away from zero instead of to even
            x = np.asarray(x, np.float64)
            r = real(x, fmt, saturate)
            a = np.abs(x)
            e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
            sp = np.ldexp(1.0, (np.maximum(e, emin) - p + 1).astype(np.int64))
            tie = np.abs(np.abs(x) / sp - np.floor(np.abs(x) / sp) - 0.5) == 0
            return np.where(tie & (a > 0), np.copysign(np.abs(r) + np.where(np.abs(r) < a, sp, 0), x), r)
        if variant == "truncate":        # drops the low bits instead of rounding
            x = np.asarray(x, np.float64)
            r = real(x, fmt, saturate)
            a = np.abs(x)
            e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
            sp = np.ldexp(1.0, (np.maximum(e, emin) - p + 1).astype(np.int64))
            t = np.copysign(np.floor(a / sp) * sp, x)
            return np.where(np.isfinite(r) & (np.abs(r) <= vmax), t, r)
        if variant == "no_subnormals":   # flushes below the smallest normal to zero
            r = real(x, fmt, saturate)
            return np.where(np.abs(r) < 2.0 ** emin, 0.0 * r, r)
        if variant == "one_bit_short":   # one significant bit too few
            return real(x, (p - 1, emin, vmax), saturate)
        if variant == "no_saturation":   # e4m3 overflow to inf
            return real(x, fmt, False)
        raise AssertionError(variant)
    return rnd


@pytest.mark.parametrize("variant", ["half_away", "truncate", "no_subnormals", "one_bit_short", "no_saturation"])
def test_readcopy_pins_catch(monkeypatch, variant):
    monkeypatch.setattr(readcopy, "round_rne", _round_mutant(variant))
    with np.errstate(all="ignore"):
        failed = _run_pins(pins_rc)
    assert failed, f"mutant {variant} passed every read-copy pin"


def test_readcopy_row_scale_mutant_caught(monkeypatch):
    """Scale by the row's mean magnitude instead of its maximum."""
    def rows(x):
        x = np.asarray(x, np.float32)
        m = np.mean(np.abs(x), axis=-1, keepdims=True).astype(np.float32)
        inv = np.where(m > 0, np.float32(448) / m, np.float32(0)).astype(np.float32)
        codes = readcopy.e4m3_bits(readcopy.to_e4m3((x * inv).astype(np.float64)))
        return codes, (m / np.float32(448)).astype(np.float32)[..., 0]
    monkeypatch.setattr(readcopy, "e4m3_rows", rows)
    failed = _run_pins(pins_rc)
    assert failed


def test_emulation_mutants_caught(monkeypatch):
    """int8 codes rounded half away from zero; a tile scale over 32 rows
    instead of 64; the scale's reciprocal taken after the product."""
    real = readcopy.emulate_quantise

    def half_away(t, fmt):
        if fmt == "int8":
            t = np.asarray(t, np.float64)
            return np.clip(np.sign(t) * np.floor(np.abs(t) + 0.5), -127.0, 127.0)
        return real(t, fmt)
    monkeypatch.setattr(readcopy, "emulate_quantise", half_away)
    assert _run_pins(pins_rc)
    monkeypatch.setattr(readcopy, "emulate_quantise", real)

    real_read = readcopy.emulate_read

    def tile32(h, fmt, scale):
        if scale != "tile64":
            return real_read(h, fmt, scale)
        h = np.asarray(h, np.float32)
        out = np.empty(h.shape)
        for i in range(0, h.shape[-2], 32):          # one scale per 32 rows
            blk = h[..., i:i + 32, :]
            m = np.max(np.abs(blk), axis=(-2, -1), keepdims=True)
            qmax = np.float32(readcopy.EMU_QMAX[fmt])
            inv = np.where(m > 0, qmax / m, np.float32(0)).astype(np.float32)
            q = readcopy.emulate_quantise((blk * inv).astype(np.float32).astype(np.float64), fmt)
            out[..., i:i + 32, :] = (q.astype(np.float32) * (m / qmax).astype(np.float32)).astype(np.float32)
        return out
    monkeypatch.setattr(readcopy, "emulate_read", tile32)
    assert _run_pins(pins_rc)
