"""Whole decode sessions on the conventional recurrence (oracle; test-only).

The expected result of a ReplaySSM run is the result of conventional decoding
over the same tokens ("ReplaySSM Caches Inputs Instead of State...", section
"How ReplaySSM works": outputs match conventional decoding up to
floating-point differences; the checkpoint is the state at the folded token).
These generators therefore advance a conventional state token by token and run
the cursor model beside it to say which sequences flushed or folded.

All arrays are numpy; records are widened to fp64 before any arithmetic.
A session over a subset of sequences is the same session restricted to them:
every sequence is independent.
"""
import numpy as np

from . import cursors as cur
from . import gdn
from . import kda
from . import mamba2


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _take(rec, j):
    """Record j of a stacked record dict (arrays [Bt, n, ...])."""
    return {k: v[:, j] for k, v in rec.items()}


def _where(mask, new, old):
    return np.where(mask.reshape(mask.shape + (1,) * (new.ndim - 1)), new, old)


# ----------------------------------------------------------------------------- Mamba-2

def _m2_step(h, r, A, D):
    return mamba2.conventional_step_layer(h, _f64(r["x"]), _f64(r["z"]), _f64(r["B"]),
                                          _f64(r["C"]), _f64(r["dt"]), _f64(A), _f64(D))


def mamba2_prefill(h0, prefill, counts, A, D):
    """Conventional state after each sequence's first counts[b] prefill records."""
    h = _f64(h0).copy()
    counts = np.asarray(counts)
    n = prefill["x"].shape[1] if prefill is not None else 0
    for j in range(n):
        mask = j < counts
        if not mask.any():
            break
        hn, _ = _m2_step(h, _take(prefill, j), A, D)
        h = _where(mask, hn, h)
    return h


def mamba2_ar_session(h0, prefill, starts, counts, steps, A, D, L):
    """AR decode. ``steps`` yields record dicts x,z [Bt,H,P], B,C [Bt,G,N], dt [Bt,H].

    Yields per step a dict: y [Bt,H,P]; flushed [Bt] bool; state [Bt,H,P,N]
    (the conventional state after the step, which a flushed sequence's
    checkpoint must equal); cursors [Bt,4]; slots [Bt] (ring slot written,
    -1 on a flush).
    """
    h = mamba2_prefill(h0, prefill, counts, A, D)
    cs = [(int(s), int(c), 0, 0) for s, c in zip(starts, counts)]
    for rec in steps:
        h, y = _m2_step(h, rec, A, D)
        flushed = np.zeros(len(cs), bool)
        slots = np.full(len(cs), -1)
        for b, c in enumerate(cs):
            nc, slot, fl, ok = cur.ar_step(c, L)
            assert ok, "the session keeps every cursor valid"
            cs[b] = nc
            flushed[b] = fl
            slots[b] = -1 if fl else slot
        yield {"y": y, "flushed": flushed, "state": h, "cursors": np.array(cs, np.int64), "slots": slots}


def mamba2_spec_session(h0, prefill, starts, counts, verifies, kepts, A, D, L):
    """Speculative decode. ``verifies`` yields record dicts with a draft axis
    (x,z [Bt,K,H,P], B,C [Bt,K,G,N], dt [Bt,K,H]); ``kepts`` yields kept [Bt].

    Output i of a verify continues conventional decoding from the committed
    state through drafts 0..i. Yields per verify a dict: y [Bt,K,H,P];
    folded [Bt]; committed_state (the state before the verify: a folded
    sequence's checkpoint must equal it); cursors_verify, cursors_commit [Bt,4].
    """
    h = mamba2_prefill(h0, prefill, counts, A, D)
    cs = [(int(s), int(c), 0, 0) for s, c in zip(starts, counts)]
    for rec, kept in zip(verifies, kepts):
        K = rec["x"].shape[1]
        committed = h
        folded = np.zeros(len(cs), bool)
        for b, c in enumerate(cs):
            nc, _, fold, ok = cur.verify(c, K, L)
            assert ok
            cs[b] = nc
            folded[b] = fold
        cv = np.array(cs, np.int64)
        hs, ys = [], []
        hi = committed
        for i in range(K):
            hi, yi = _m2_step(hi, _take(rec, i), A, D)
            hs.append(hi)
            ys.append(yi)
        y = np.stack(ys, axis=1)
        kept = np.asarray(kept)
        h = committed.copy()
        for b in range(len(cs)):
            if kept[b] > 0:
                h[b] = hs[kept[b] - 1][b]
            nc, ok = cur.commit(cs[b], int(kept[b]), L)
            assert ok
            cs[b] = nc
        yield {"y": y, "folded": folded, "committed_state": committed,
               "cursors_verify": cv, "cursors_commit": np.array(cs, np.int64), "state": h}


def mamba2_flush_expected(h0, ring_window, A):
    """Standalone flush: fold each sequence's window into its checkpoint.
    ring_window: list over sequences of (xs [m,H,P], Bs [m,G,N], dts [m,H])."""
    out = _f64(h0).copy()
    for b, (xs, Bs, dts) in enumerate(ring_window):
        m = xs.shape[0]
        if m == 0:
            continue
        hb = out[b]
        for k in range(m):
            r = {"x": xs[None, k], "z": np.zeros_like(xs[None, k]), "B": Bs[None, k],
                 "C": np.zeros_like(Bs[None, k]), "dt": dts[None, k]}
            hb, _ = _m2_step(hb[None], r, A, np.zeros_like(_f64(A)))
            hb = hb[0]
        out[b] = hb
    return out


# ----------------------------------------------------------------------------- Gated DeltaNet

def _gdn_step(S, r):
    return gdn.conventional_step(S, _f64(r["q"]), _f64(r["k"]), _f64(r["v"]), _f64(r["g"]), _f64(r["beta"]))


def gdn_prefill(S0, prefill, counts):
    S = _f64(S0).copy()
    counts = np.asarray(counts)
    n = prefill["q"].shape[1] if prefill is not None else 0
    for j in range(n):
        mask = j < counts
        if not mask.any():
            break
        Sn, _ = _gdn_step(S, _take(prefill, j))
        S = _where(mask, Sn, S)
    return S


def gdn_ar_session(S0, prefill, starts, counts, steps, L):
    """AR decode for Gated DeltaNet; records q,k [Bt,H,dk], v [Bt,H,dv], g,beta [Bt,H].
    Yields dicts like mamba2_ar_session with o [Bt,H,dv] in place of y."""
    S = gdn_prefill(S0, prefill, counts)
    cs = [(int(s), int(c), 0, 0) for s, c in zip(starts, counts)]
    for rec in steps:
        S, o = _gdn_step(S, rec)
        flushed = np.zeros(len(cs), bool)
        for b, c in enumerate(cs):
            nc, slot, fl, ok = cur.ar_step(c, L)
            assert ok
            cs[b] = nc
            flushed[b] = fl
        yield {"o": o, "flushed": flushed, "state": S, "cursors": np.array(cs, np.int64)}


def gdn_spec_session(S0, prefill, starts, counts, verifies, kepts, L):
    """Speculative decode for Gated DeltaNet ("ReplaySSM", introduction:
    drafts verified output-only, rejected ones dropped by moving a pointer).
    ``verifies`` yields record dicts with a draft axis (q,k [Bt,K,H,dk],
    v [Bt,K,H,dv], g,beta [Bt,K,H]); ``kepts`` yields kept [Bt].

    Output i of a verify continues conventional decoding from the committed
    state through drafts 0..i. Yields per verify a dict: o [Bt,K,H,dv];
    folded [Bt]; committed_state (the state before the verify: a folded
    sequence's checkpoint must equal it); cursors_verify, cursors_commit
    [Bt,4]; state (the committed state after the commit).
    """
    return _delta_spec_session(_gdn_step, gdn_prefill(S0, prefill, counts), starts, counts, verifies, kepts, L)


def _delta_spec_session(step, S, starts, counts, verifies, kepts, L):
    """The speculative session of a delta-rule layer, from the committed state S."""
    cs = [(int(s), int(c), 0, 0) for s, c in zip(starts, counts)]
    for rec, kept in zip(verifies, kepts):
        K = rec["q"].shape[1]
        committed = S
        folded = np.zeros(len(cs), bool)
        for b, c in enumerate(cs):
            nc, _, fold, ok = cur.verify(c, K, L)
            assert ok
            cs[b] = nc
            folded[b] = fold
        cv = np.array(cs, np.int64)
        Ss, os_ = [], []
        Si = committed
        for i in range(K):
            Si, oi = step(Si, _take(rec, i))
            Ss.append(Si)
            os_.append(oi)
        o = np.stack(os_, axis=1)
        kept = np.asarray(kept)
        S = committed.copy()
        for b in range(len(cs)):
            if kept[b] > 0:
                S[b] = Ss[kept[b] - 1][b]
            nc, ok = cur.commit(cs[b], int(kept[b]), L)
            assert ok
            cs[b] = nc
        yield {"o": o, "folded": folded, "committed_state": committed,
               "cursors_verify": cv, "cursors_commit": np.array(cs, np.int64), "state": S}


# ----------------------------------------------------------------------------- Kimi Delta Attention

def _kda_step(S, r):
    return kda.conventional_step(S, _f64(r["q"]), _f64(r["k"]), _f64(r["v"]), _f64(r["g"]), _f64(r["beta"]))


def kda_prefill(S0, prefill, counts):
    S = _f64(S0).copy()
    counts = np.asarray(counts)
    n = prefill["q"].shape[1] if prefill is not None else 0
    for j in range(n):
        mask = j < counts
        if not mask.any():
            break
        Sn, _ = _kda_step(S, _take(prefill, j))
        S = _where(mask, Sn, S)
    return S


def kda_ar_session(S0, prefill, starts, counts, steps, L):
    """AR decode for Kimi Delta Attention; records q,k,g [Bt,H,dk], v [Bt,H,dv],
    beta [Bt,H]. Yields dicts like gdn_ar_session."""
    S = kda_prefill(S0, prefill, counts)
    cs = [(int(s), int(c), 0, 0) for s, c in zip(starts, counts)]
    for rec in steps:
        S, o = _kda_step(S, rec)
        flushed = np.zeros(len(cs), bool)
        for b, c in enumerate(cs):
            nc, slot, fl, ok = cur.ar_step(c, L)
            assert ok
            cs[b] = nc
            flushed[b] = fl
        yield {"o": o, "flushed": flushed, "state": S, "cursors": np.array(cs, np.int64)}


def kda_spec_session(S0, prefill, starts, counts, verifies, kepts, L):
    """Speculative decode for Kimi Delta Attention: as gdn_spec_session, with
    g [Bt,K,H,dk] one log decay per key channel."""
    return _delta_spec_session(_kda_step, kda_prefill(S0, prefill, counts), starts, counts, verifies, kepts, L)
