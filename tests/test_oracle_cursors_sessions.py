"""Pins for the cursor model (hand-derived traces, invariants) and for the
session runners (speculative decode with every draft kept equals AR decode;
with drafts rejected it equals AR decode over the kept prefix)."""
import numpy as np
import pytest

from oracle import cursors as cur
from oracle import gdn, kda, mamba2, sessions


def test_ar_trace_by_hand():
    L = 4
    c = (1, 2, 0, 0)
    c, slot, fl, ok = cur.ar_step(c, L)
    assert (c, slot, fl, ok) == ((1, 3, 0, 0), 3, False, True)
    c, slot, fl, ok = cur.ar_step(c, L)      # 4th record: flush, slot (1+3)%4 = 0
    assert (c, slot, fl, ok) == ((1, 0, 0, 0), 0, True, True)
    c, slot, fl, ok = cur.ar_step(c, L)
    assert (c, slot, fl, ok) == ((1, 1, 0, 0), 1, False, True)


def test_ar_L1_flushes_every_step():
    c = (0, 0, 0, 0)
    for _ in range(5):
        c, slot, fl, ok = cur.ar_step(c, 1)
        assert ok and fl and c == (0, 0, 0, 0)


def test_spec_trace_by_hand():
    L, K = 4, 3
    c = (2, 1, 0, 0)
    c, slots, fold, ok = cur.verify(c, K, L)        # 1 + 3 = 4, not > 4: no fold
    assert (c, slots, fold, ok) == ((2, 1, 3, 0), [3, 0, 1], False, True)
    c, ok = cur.commit(c, 2, L)
    assert (c, ok) == ((2, 3, 0, 0), True)
    c, slots, fold, ok = cur.verify(c, K, L)        # 3 + 3 > 4: fold the 3 committed
    assert (c, slots, fold, ok) == ((2, 3, 3, cur.FOLDED), [1, 2, 3], True, True)
    c, ok = cur.commit(c, 1, L)                     # start = (2+3)%4 = 1, count = 1
    assert (c, ok) == ((1, 1, 0, 0), True)
    # the next record lands right after the kept draft (which sat at slot 1)
    assert cur.verify(c, K, L)[1][0] == 2


def test_error_cases_leave_cursor_unchanged():
    L = 4
    assert cur.ar_step((0, 4, 0, 0), L)[3] is False          # full window
    assert cur.ar_step((0, 1, 2, 0), L)[3] is False          # uncommitted drafts
    assert cur.ar_step((4, 0, 0, 0), L)[3] is False          # start out of range
    assert cur.verify((0, 1, 3, 0), 3, L)[3] is False        # verify twice
    assert cur.verify((0, 1, 0, 0), 5, L)[3] is False        # K > L
    assert cur.commit((0, 1, 3, 0), 4, L) == ((0, 1, 3, 0), False)   # kept > pending
    assert cur.commit((0, 1, 0, 0), 0, L) == ((0, 1, 0, 0), True)    # idle sequence
    assert cur.flush((0, 2, 1, 0), L)[2] is False
    assert cur.flush((3, 2, 0, 0), L) == ((1, 0, 0, 0), 2, True)


def test_random_spec_invariants():
    rng = np.random.default_rng(7)
    for L in (1, 4, 16, 32):
        for K in sorted({1, min(4, L), L}):
            c = (int(rng.integers(L)), int(rng.integers(L + 1)), 0, 0)
            for _ in range(300):
                start, count = c[0], c[1]
                window = {(start + j) % L for j in range(count)}
                nc, slots, fold, ok = cur.verify(c, K, L)
                assert ok
                if not fold:
                    assert not window & set(slots)      # drafts never overwrite committed records
                    assert count + K <= L
                assert len(set(slots)) == K
                kept = int(rng.integers(K + 1))
                c2, ok = cur.commit(nc, kept, L)
                assert ok and 0 <= c2[1] <= L and c2[2] == 0
                if fold and kept:
                    assert c2[0] == slots[0]             # new window starts at draft 0
                c = c2


def _records(rng, Bt, H, P, N, G, n):
    return {"x": rng.standard_normal((Bt, n, H, P)), "z": rng.standard_normal((Bt, n, H, P)),
            "B": rng.standard_normal((Bt, n, G, N)) / np.sqrt(N), "C": rng.standard_normal((Bt, n, G, N)) / np.sqrt(N),
            "dt": np.log1p(np.exp(rng.normal(-2, 0.5, (Bt, n, H))))}


@pytest.mark.parametrize("reject", [False, True])
def test_spec_session_matches_ar(rng, reject):
    """Spec decode with kept drafts equals AR decode over exactly the kept tokens."""
    Bt, H, P, N, G, L, K, V = 3, 4, 3, 5, 2, 6, 3, 7
    A, D = -np.exp(rng.uniform(0, 2.5, H)), rng.standard_normal(H)
    h0 = 0.1 * rng.standard_normal((Bt, H, P, N))
    drafts = [_records(rng, Bt, H, P, N, G, K) for _ in range(V)]
    kepts = [rng.integers(1, K + 1, Bt) if reject else np.full(Bt, K) for _ in range(V)]
    starts, counts = np.array([0, 2, 5]), np.zeros(Bt, int)
    spec = list(sessions.mamba2_spec_session(h0, None, starts, counts, drafts, kepts, A, D, L))
    for b in range(Bt):
        # AR over the kept tokens of sequence b, in order
        toks = [(v, i) for v in range(V) for i in range(kepts[v][b])]
        h = h0[b:b + 1]
        for (v, i) in toks:
            r = {k: a[b:b + 1, i] for k, a in drafts[v].items()}
            h, y = mamba2.conventional_step_layer(h, r["x"], r["z"], r["B"], r["C"], r["dt"], A, D)
            np.testing.assert_allclose(spec[v]["y"][b, i], y[0], rtol=1e-12, atol=1e-14)
            if i == kepts[v][b] - 1:
                np.testing.assert_allclose(spec[v]["state"][b], h[0], rtol=1e-12, atol=1e-14)
        # the cursor count equals the kept tokens since the last fold
        c = spec[-1]["cursors_commit"][b]
        assert 0 <= c[1] <= L and c[2] == 0


def test_ar_session_flush_trace(rng):
    """AR session: flushes land exactly every L steps after the prefill count."""
    Bt, H, P, N, G, L = 4, 2, 3, 4, 1, 5
    A, D = -np.exp(rng.uniform(0, 2.5, H)), rng.standard_normal(H)
    counts, starts = np.array([0, 1, 3, 4]), np.array([0, 3, 4, 1])
    pre = _records(rng, Bt, H, P, N, G, L - 1)
    steps = [{k: a[:, 0] for k, a in _records(rng, Bt, H, P, N, G, 1).items()} for _ in range(12)]
    out = list(sessions.mamba2_ar_session(0.1 * rng.standard_normal((Bt, H, P, N)), pre, starts, counts, steps, A, D, L))
    for b in range(Bt):
        fl = [t for t in range(12) if out[t]["flushed"][b]]
        first = L - counts[b] - 1
        assert fl == list(range(first, 12, L))


def test_flush_expected_equals_replay(rng):
    Bt, H, P, N, G = 2, 4, 3, 5, 2
    A = -np.exp(rng.uniform(0, 2.5, H))
    h0 = rng.standard_normal((Bt, H, P, N))
    win = []
    for b, m in enumerate([3, 0]):
        win.append((rng.standard_normal((m, H, P)), rng.standard_normal((m, G, N)), rng.uniform(0.05, 0.5, (m, H))))
    out = sessions.mamba2_flush_expected(h0, win, A)
    xs, Bs, dts = win[0]
    Bh = Bs[:, mamba2.group_of_head(H, G)]
    ref = mamba2.replay_state(h0[0], np.moveaxis(xs, 0, 1), np.moveaxis(Bh, 0, 1), np.moveaxis(dts, 0, 1), A)
    np.testing.assert_allclose(out[0], ref, rtol=1e-12)
    np.testing.assert_array_equal(out[1], h0[1])


def _gdn_records(rng, Bt, H, dk, dv, n):
    q = rng.standard_normal((Bt, n, H, dk))
    k = rng.standard_normal((Bt, n, H, dk))
    return {"q": q / np.linalg.norm(q, axis=-1, keepdims=True), "k": k / np.linalg.norm(k, axis=-1, keepdims=True),
            "v": rng.standard_normal((Bt, n, H, dv)), "g": -np.log1p(np.exp(rng.standard_normal((Bt, n, H)))),
            "beta": 1 / (1 + np.exp(-rng.standard_normal((Bt, n, H))))}


@pytest.mark.parametrize("reject", [False, True])
def test_gdn_spec_session_matches_ar(rng, reject):
    """GDN spec decode with kept drafts equals AR decode over exactly the kept
    tokens (outputs, committed state); cursors follow the verify/commit rules."""
    Bt, H, dk, dv, L, K, V = 3, 2, 4, 3, 6, 3, 7
    S0 = 0.1 * rng.standard_normal((Bt, H, dv, dk))
    drafts = [_gdn_records(rng, Bt, H, dk, dv, K) for _ in range(V)]
    kepts = [rng.integers(1, K + 1, Bt) if reject else np.full(Bt, K) for _ in range(V)]
    starts, counts = np.array([0, 2, 5]), np.zeros(Bt, int)
    spec = list(sessions.gdn_spec_session(S0, None, starts, counts, drafts, kepts, L))
    for b in range(Bt):
        S = S0[b:b + 1]
        for v in range(V):
            for i in range(kepts[v][b]):
                r = {k: a[b:b + 1, i] for k, a in drafts[v].items()}
                S, o = gdn.conventional_step(S, r["q"], r["k"], r["v"], r["g"], r["beta"])
                np.testing.assert_allclose(spec[v]["o"][b, i], o[0], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(spec[v]["state"][b], S[0], rtol=1e-12, atol=1e-14)
        c = spec[-1]["cursors_commit"][b]
        assert 0 <= c[1] <= L and c[2] == 0
    # a rejected draft's output is still the continuation through it
    v, b = 0, 0
    S = S0[b:b + 1]
    for i in range(K):
        r = {k: a[b:b + 1, i] for k, a in drafts[v].items()}
        S, o = gdn.conventional_step(S, r["q"], r["k"], r["v"], r["g"], r["beta"])
        np.testing.assert_allclose(spec[v]["o"][b, i], o[0], rtol=1e-12, atol=1e-14)


def test_gdn_spec_session_folds_like_mamba2(rng):
    """The fold flags and cursor trace depend only on the cursor rules: the
    GDN and Mamba-2 sessions agree on them for the same kept counts."""
    Bt, L, K, V = 4, 5, 3, 9
    starts, counts = np.array([0, 1, 4, 2]), np.array([0, 3, 4, 1])
    kepts = [rng.integers(1, K + 1, Bt) for _ in range(V)]
    g = list(sessions.gdn_spec_session(np.zeros((Bt, 1, 2, 2)), _gdn_records(rng, Bt, 1, 2, 2, L - 1), starts, counts,
                                       [_gdn_records(rng, Bt, 1, 2, 2, K) for _ in range(V)], kepts, L))
    m = list(sessions.mamba2_spec_session(np.zeros((Bt, 1, 2, 2)), _records(rng, Bt, 1, 2, 2, 1, L - 1), starts, counts,
                                          [_records(rng, Bt, 1, 2, 2, 1, K) for _ in range(V)], kepts,
                                          -np.ones(1), np.zeros(1), L))
    for a, c in zip(g, m):
        np.testing.assert_array_equal(a["folded"], c["folded"])
        np.testing.assert_array_equal(a["cursors_verify"], c["cursors_verify"])
        np.testing.assert_array_equal(a["cursors_commit"], c["cursors_commit"])
    assert any(x["folded"].any() for x in g)


def _kda_records(rng, Bt, H, dk, dv, n):
    r = _gdn_records(rng, Bt, H, dk, dv, n)
    r["g"] = -0.5 * np.log1p(np.exp(rng.standard_normal((Bt, n, H, dk))))  # one decay per key channel
    return r


@pytest.mark.parametrize("reject", [False, True])
def test_kda_spec_session_matches_ar(rng, reject):
    """KDA spec decode with kept drafts equals AR decode over exactly the kept
    tokens (outputs, committed state), from prefilled windows; a rejected
    draft's output is the continuation through it."""
    Bt, H, dk, dv, L, K, V = 3, 2, 4, 3, 6, 3, 7
    S0 = 0.1 * rng.standard_normal((Bt, H, dv, dk))
    pre = _kda_records(rng, Bt, H, dk, dv, L - 1)
    starts, counts = np.array([0, 2, 5]), np.array([0, 3, 5])
    drafts = [_kda_records(rng, Bt, H, dk, dv, K) for _ in range(V)]
    kepts = [rng.integers(1, K + 1, Bt) if reject else np.full(Bt, K) for _ in range(V)]
    spec = list(sessions.kda_spec_session(S0, pre, starts, counts, drafts, kepts, L))
    for b in range(Bt):
        S = S0[b:b + 1]
        for j in range(counts[b]):
            r = {k: a[b:b + 1, j] for k, a in pre.items()}
            S, _ = kda.conventional_step(S, r["q"], r["k"], r["v"], r["g"], r["beta"])
        for v in range(V):
            Sv = S
            for i in range(K):
                r = {k: a[b:b + 1, i] for k, a in drafts[v].items()}
                Sv, o = kda.conventional_step(Sv, r["q"], r["k"], r["v"], r["g"], r["beta"])
                np.testing.assert_allclose(spec[v]["o"][b, i], o[0], rtol=1e-12, atol=1e-14)
                if i + 1 == kepts[v][b]:
                    Snext = Sv
            S = Snext
            np.testing.assert_allclose(spec[v]["state"][b], S[0], rtol=1e-12, atol=1e-14)
    assert any(x["folded"].any() for x in spec)
