"""Kimi Delta Attention parity on the GPU, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import harness as H
from oracle import kda as ok
from oracle import sessions
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import KDAWorkload as KW
from recurrent_state_decode_gb300.state import KDAState, kda_from_workload

pytestmark = pytest.mark.gpu

TOL_Y32, TOL_CKPT, TOL_BF16_EXCESS = 1e-4, 1e-5, 2e-3


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def run_kda(w, out_dtype=bd.RSSM_F32, seqs=None, steps=None):
    dev = "cuda"
    st, pre, starts, counts = kda_from_workload(w, dev, out_dtype)
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    feed = H.Feed()
    sess = sessions.kda_ar_session(H.F64(st.S[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                   counts[seqs].cpu().numpy(), feed, w.buf_len)
    o = st.new_output()
    flushes = 0
    for t in range(w.steps if steps is None else steps):
        rec = I.kda_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, seqs)
        st.step(rec, o)
        exp = next(sess)
        og_ = H.F64(o[seqs])
        if out_dtype == bd.RSSM_F32:
            err = H.rel_l2(og_, exp["o"])
            assert err <= TOL_Y32, (t, err)
        else:
            ex = H.bf16_excess(og_, exp["o"])
            assert ex <= TOL_BF16_EXCESS, (t, ex)
        np.testing.assert_array_equal(st.cursors[seqs].cpu().numpy(), exp["cursors"])
        for i, b in enumerate(seqs):
            if exp["flushed"][i]:
                flushes += 1
                e = H.rel_l2(H.F64(st.S[b]), exp["state"][i])
                assert e <= TOL_CKPT, (t, b, e)
    assert H.status(st) == 0
    return flushes


KSHAPES = [
    KW("kda_128", 2, 4, 128, 128, 16, 34, seed=401),            # the serving tile
    KW("kda_L1", 2, 3, 128, 128, 1, 6, seed=402),               # every step flushes
    KW("kda_L5", 3, 2, 128, 128, 5, 23, seed=403),              # ragged window, wraps often
    KW("kda_L31", 2, 2, 128, 128, 31, 70, seed=404),            # longest window of the step kernel
    KW("kda_H3", 3, 3, 128, 128, 7, 20, seed=405),              # odd head count
    KW("kda_cold", 4, 2, 128, 128, 8, 20, seed=406, zero_ckpt=True, prefill=False),  # empty windows, zero state
]


@pytest.mark.parametrize("w", KSHAPES, ids=lambda w: w.name)
@pytest.mark.parametrize("out", [bd.RSSM_F32, bd.RSSM_BF16], ids=["f32", "bf16"])
def test_kda_shapes(w, out):
    assert run_kda(w, out) > 0


def test_kda_strong_decays():
    """Per-token decays down to exp(-12) on some channels: the window factors
    are exponentials of later-minus-earlier sums only, so nothing overflows."""
    w = KW("kda_strong", 2, 2, 128, 128, 16, 20, seed=407)
    dev = "cuda"
    st, pre, starts, counts = kda_from_workload(w, dev)
    feed = H.Feed()
    sess = sessions.kda_ar_session(H.F64(st.S), H.sub(pre, slice(None)), starts.cpu().numpy(), counts.cpu().numpy(),
                                   feed, w.buf_len)
    o = st.new_output()
    for t in range(w.steps):
        rec = I.kda_step_inputs(w, t, dev)
        rec["g"] = rec["g"] * 4.0  # down to about -12
        feed.rec = H.sub(rec, slice(None))
        st.step(rec, o)
        exp = next(sess)
        assert torch.isfinite(o).all()
        assert H.rel_l2(H.F64(o), exp["o"]) <= TOL_Y32, t
        for b in range(w.batch):
            if exp["flushed"][b]:
                assert H.rel_l2(H.F64(st.S[b]), exp["state"][b]) <= TOL_CKPT
    assert H.status(st) == 0


@pytest.mark.parametrize("shape", [(40, 24), (128, 128), (256, 256)], ids=["ragged", "128", "256"])
def test_kda_conventional_kernel(shape):
    dk, dv = shape
    w = KW("kconv", 3, 3, dk, dv, 16, 12, seed=408)
    dev = "cuda"
    S = I.gdn_checkpoint(w, dev)
    Sh = H.F64(S)
    o = torch.empty((w.batch, w.nheads, w.dv), device=dev)
    desc = bd.kda_desc(w.batch, w.nheads, w.dk, w.dv, w.buf_len)
    for t in range(w.steps):
        rec = I.kda_step_inputs(w, t, dev)
        bd.check(bd.rssm_kda_conventional_step(desc, S, rec["q"], rec["k"], rec["v"], rec["g"], rec["beta"], o))
        r = {k: H.F64(v) for k, v in rec.items()}
        Sh, oe = ok.conventional_step(Sh, r["q"], r["k"], r["v"], r["g"], r["beta"])
        assert H.rel_l2(H.F64(o), oe) <= TOL_Y32
        assert H.rel_l2(H.F64(S), Sh) <= TOL_CKPT


def test_kda_standalone_flush():
    w = KW("kflush", 3, 2, 128, 128, 8, 5, seed=409)
    dev = "cuda"
    st, pre, starts, counts = kda_from_workload(w, dev)
    feed = H.Feed()
    sess = sessions.kda_ar_session(H.F64(st.S), H.sub(pre, slice(None)), starts.cpu().numpy(), counts.cpu().numpy(),
                                   feed, w.buf_len)
    o = st.new_output()
    for t in range(w.steps):
        rec = I.kda_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, slice(None))
        st.step(rec, o)
        exp = next(sess)
    before = st.cursors.cpu().numpy()
    st.flush()
    cur = st.cursors.cpu().numpy()
    np.testing.assert_array_equal(cur[:, 0], (before[:, 0] + before[:, 1]) % w.buf_len)
    np.testing.assert_array_equal(cur[:, 1:], 0)
    for b in range(w.batch):
        assert H.rel_l2(H.F64(st.S[b]), exp["state"][b]) <= TOL_CKPT
    assert H.status(st) == 0


@pytest.mark.parametrize("w", [KW("kprime", 3, 2, 128, 128, 16, 1, seed=410),
                               KW("kprime_L32", 2, 2, 128, 128, 32, 1, seed=411)], ids=lambda w: w.name)
def test_kda_prime_matches_window_corrections(w):
    """rssm_kda_prime fills ring.e with each window record's correction e_t,
    checked against the oracle's forward substitution (L = 32 included: the
    prime and the flush take every window length)."""
    st, pre, starts, counts = kda_from_workload(w, "cuda")  # places the windows, then primes
    S0 = H.F64(st.S)
    re = H.F64(st.re)
    checked = 0
    for b in range(w.batch):
        c, s0 = int(counts[b]), int(starts[b])
        if c == 0:
            continue
        r = {k: H.F64(v[b, :c]) for k, v in pre.items()}  # [c, H, ...]
        ks, vs, gs = np.moveaxis(r["k"], 0, 1), np.moveaxis(r["v"], 0, 1), np.moveaxis(r["g"], 0, 1)
        bs = r["beta"].T
        e = ok.replay_corrections(S0[b], ks, vs, gs, bs)  # [H, c, dv]
        slots = [(s0 + t) % w.buf_len for t in range(c)]
        assert H.rel_l2(re[b][:, slots], e) <= 1e-5
        checked += 1
    assert checked > 0
    assert H.status(st) == 0


def test_kda_device_errors_skip_sequence():
    """Bad cursors are reported, left as they were and skipped; the other sequences step."""
    w = KW("kerr", 3, 2, 128, 128, 4, 1, seed=412, prefill=False)
    dev = "cuda"
    st, _, _, _ = kda_from_workload(w, dev)
    st.cursors[1] = torch.tensor([0, 7, 0, 0], dtype=torch.int32)  # count > L
    st.cursors[2] = torch.tensor([0, 1, 2, 0], dtype=torch.int32)  # uncommitted drafts
    before = st.cursors.clone()
    S0 = st.S.clone()
    re0 = st.re.clone()
    o = st.new_output().fill_(float("nan"))
    st.step(I.kda_step_inputs(w, 0, dev), o)
    torch.cuda.synchronize()
    assert H.status(st) in (bd.RSSM_DEV_BAD_CURSOR, bd.RSSM_DEV_PENDING)
    assert torch.isfinite(o[0]).all()
    assert torch.isnan(o[1:]).all()
    assert torch.equal(st.cursors[1:], before[1:])
    assert st.cursors[0].tolist() == [0, 1, 0, 0]
    assert torch.equal(st.S[1:], S0[1:])
    assert torch.equal(st.re[1:], re0[1:])


def test_kda_unsupported_shapes():
    st = KDAState(2, 2, 64, 128, 8)
    rec = {k: torch.zeros(1, device="cuda") for k in ("q", "k", "v", "g", "beta")}
    assert bd.rssm_kda_step(st.desc, st.S, st.ring, st.cursors, rec["q"], rec["k"], rec["v"], rec["g"],
                            rec["beta"], st.S) == bd.RSSM_ERR_UNSUPPORTED
    assert bd.rssm_kda_flush(st.desc, st.S, st.ring, st.cursors) == bd.RSSM_ERR_UNSUPPORTED
    st32 = KDAState(2, 2, 128, 128, 32)
    assert bd.rssm_kda_step(st32.desc, st32.S, st32.ring, st32.cursors, rec["q"], rec["k"], rec["v"], rec["g"],
                            rec["beta"], st32.S) == bd.RSSM_ERR_UNSUPPORTED  # the step needs L <= 31


def test_kda_step_with_slots_matches_the_plain_call():
    w = KW("kslots", 3, 2, 128, 128, 8, 12, seed=413)
    dev = "cuda"
    sa, _, _, _ = kda_from_workload(w, dev)
    ss = KDAState(7, w.nheads, w.dk, w.dv, w.buf_len, dev)
    perm, row_of, pad = [5, 0, 3], [2, 4, 1], [0, 3]
    fields = ("S", "rq", "rk", "rv", "rg", "rbeta", "re", "cursors")
    for f in fields:
        getattr(ss, f)[perm] = getattr(sa, f)
    slots = torch.full((5,), -1, dtype=torch.int32, device=dev)
    slots[row_of] = torch.tensor(perm, dtype=torch.int32, device=dev)
    for t in range(w.steps):
        rec = I.kda_step_inputs(w, t, dev)
        oa = sa.new_output()
        sa.step(rec, oa)
        rows = {k: v[[0] * 5].clone() for k, v in rec.items()}
        for k, v in rec.items():
            rows[k][row_of] = v
        os_ = torch.full((5, w.nheads, w.dv), float("nan"), device=dev)
        ss.step(rows, os_, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(os_[row_of], oa), t
        assert torch.isnan(os_[pad]).all(), t
    for f in fields:
        assert torch.equal(getattr(ss, f)[perm], getattr(sa, f)), f
    assert H.status(sa) == 0 and H.status(ss) == 0


def test_kda_verify_commit_with_slots_matches_the_plain_calls():
    """The verify and commit through a slot table (a permuted batch with
    padding rows) give the plain calls' outputs, states, rings and cursors bit
    for bit; padding rows' outputs stay unwritten."""
    w = KW("kslots_spec", 3, 2, 128, 128, 8, 8, seed=414, drafts=3)
    dev = "cuda"
    sa, _, _, _ = kda_from_workload(w, dev)
    ss = KDAState(7, w.nheads, w.dk, w.dv, w.buf_len, dev)
    perm, row_of, pad = [5, 0, 3], [2, 4, 1], [0, 3]
    fields = ("S", "rq", "rk", "rv", "rg", "rbeta", "re", "cursors")
    for f in fields:
        getattr(ss, f)[perm] = getattr(sa, f)
    slots = torch.full((5,), -1, dtype=torch.int32, device=dev)
    slots[row_of] = torch.tensor(perm, dtype=torch.int32, device=dev)
    for t in range(w.steps):
        rec = I.kda_verify_inputs(w, t, dev)
        kept = I.accepted_kept(w, t, dev)
        oa = sa.new_verify_output(w.n_new)
        sa.verify(rec, oa)
        sa.commit(kept)
        rows = {k: v[[0] * 5].clone() for k, v in rec.items()}
        for k, v in rec.items():
            rows[k][row_of] = v
        os_ = torch.full((5, w.n_new, w.nheads, w.dv), float("nan"), device=dev)
        ss.verify(rows, os_, slots=slots)
        kept_rows = torch.full((5,), 999, dtype=torch.int32, device=dev)
        kept_rows[row_of] = kept
        ss.commit(kept_rows, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(os_[row_of], oa), t
        assert torch.isnan(os_[pad]).all(), t
    for f in fields:
        assert torch.equal(getattr(ss, f)[perm], getattr(sa, f)), f
    assert H.status(sa) == 0 and H.status(ss) == 0


# ----------------------------------------------------------------------------- speculative verify

def run_kda_spec(w, out_dtype=bd.RSSM_F32):
    dev = "cuda"
    st, pre, starts, counts = kda_from_workload(w, dev, out_dtype)
    fv, fk = H.Feed(), H.Feed()
    sess = sessions.kda_spec_session(H.F64(st.S), H.sub(pre, slice(None)), starts.cpu().numpy(),
                                     counts.cpu().numpy(), fv, fk, w.buf_len)
    o = st.new_verify_output(w.n_new)
    folds = 0
    for t in range(w.steps):
        rec = I.kda_verify_inputs(w, t, dev)
        kept = I.accepted_kept(w, t, dev)
        fv.rec = H.sub(rec, slice(None))
        fk.rec = kept.cpu().numpy()
        st.verify(rec, o)
        cv = st.cursors.cpu().numpy()
        st.commit(kept)
        exp = next(sess)
        og_ = H.F64(o)
        if out_dtype == bd.RSSM_F32:
            assert H.rel_l2(og_, exp["o"]) <= TOL_Y32, t
        else:
            assert H.bf16_excess(og_, exp["o"]) <= TOL_BF16_EXCESS, t
        np.testing.assert_array_equal(cv, exp["cursors_verify"])
        np.testing.assert_array_equal(st.cursors.cpu().numpy(), exp["cursors_commit"])
        for b in range(w.batch):
            if exp["folded"][b]:
                folds += 1
                assert H.rel_l2(H.F64(st.S[b]), exp["committed_state"][b]) <= TOL_CKPT, (t, b)
    assert H.status(st) == 0
    # the ring's cached corrections of the committed window agree with the
    # checkpoint and the window's records (what the AR step relies on)
    S, cur = H.F64(st.S), st.cursors.cpu().numpy()
    ring = {f: H.F64(getattr(st, n)) for f, n in (("k", "rk"), ("v", "rv"), ("g", "rg"), ("e", "re"))}
    beta = H.F64(st.rbeta)
    for b in range(w.batch):
        s0, c = int(cur[b, 0]), int(cur[b, 1])
        if c == 0:
            continue
        slots = [(s0 + t) % w.buf_len for t in range(c)]
        e = ok.replay_corrections(S[b], ring["k"][b][:, slots], ring["v"][b][:, slots], ring["g"][b][:, slots],
                                  beta[b][:, slots])
        assert H.rel_l2(ring["e"][b][:, slots], e) <= 1e-5, b
    return folds


KSPEC = [
    KW("kspec_128", 3, 4, 128, 128, 16, 24, seed=420, drafts=3),     # the serving tile
    KW("kspec_L5", 2, 2, 128, 128, 5, 14, seed=421, drafts=3),       # folds often
    KW("kspec_K1", 2, 2, 128, 128, 8, 12, seed=422, drafts=0),       # one record per verify
    KW("kspec_K2", 3, 2, 128, 128, 8, 12, seed=423, drafts=1),
    KW("kspec_L28", 2, 2, 128, 128, 28, 24, seed=424, drafts=3),     # L + K = 32, the longest view
    KW("kspec_K_eq_L", 3, 2, 128, 128, 4, 8, seed=425, drafts=3),    # K = L: every verify with count > 0 folds
]


@pytest.mark.parametrize("w", KSPEC, ids=lambda w: w.name)
def test_kda_spec(w):
    assert run_kda_spec(w) > 0 or w.name == "kspec_K1"


def test_kda_spec_bf16_out():
    run_kda_spec(KSPEC[0], out_dtype=bd.RSSM_BF16)


def test_kda_spec_strong_decays():
    """Speculative decode with per-token decays down to about exp(-12) per
    channel (the window, the new records and the fold): every decay factor is
    an exponential of a later-minus-earlier sum, so nothing overflows and the
    outputs, corrections and folded checkpoints stay at the fp32 tolerances."""
    w = KW("kspec_strong", 3, 2, 128, 128, 8, 16, seed=427, drafts=3)
    dev = "cuda"
    st, pre, starts, counts = kda_from_workload(w, dev)
    fv, fk = H.Feed(), H.Feed()
    sess = sessions.kda_spec_session(H.F64(st.S), H.sub(pre, slice(None)), starts.cpu().numpy(),
                                     counts.cpu().numpy(), fv, fk, w.buf_len)
    o = st.new_verify_output(w.n_new)
    folds = 0
    for t in range(w.steps):
        rec = I.kda_verify_inputs(w, t, dev)
        rec["g"] = (rec["g"] * 4.0).contiguous()
        kept = I.accepted_kept(w, t, dev)
        fv.rec, fk.rec = H.sub(rec, slice(None)), kept.cpu().numpy()
        st.verify(rec, o)
        st.commit(kept)
        exp = next(sess)
        assert torch.isfinite(o).all()
        assert H.rel_l2(H.F64(o), exp["o"]) <= TOL_Y32, t
        for b in range(w.batch):
            if exp["folded"][b]:
                folds += 1
                assert H.rel_l2(H.F64(st.S[b]), exp["committed_state"][b]) <= TOL_CKPT, (t, b)
    assert folds > 0
    assert H.status(st) == 0


def test_kda_spec_unsupported_and_invalid():
    st = KDAState(2, 2, 128, 128, 30)
    rec = {k: torch.zeros(1, device="cuda") for k in ("q", "k", "v", "g", "beta")}
    args = (st.S, st.ring, st.cursors, rec["q"], rec["k"], rec["v"], rec["g"], rec["beta"], st.S)
    assert bd.rssm_kda_spec_verify(st.desc, 3, *args) == bd.RSSM_ERR_UNSUPPORTED   # L + K > 32
    st8 = KDAState(2, 2, 128, 128, 8)
    args8 = (st8.S, st8.ring, st8.cursors, rec["q"], rec["k"], rec["v"], rec["g"], rec["beta"], st8.S)
    assert bd.rssm_kda_spec_verify(st8.desc, 5, *args8) == bd.RSSM_ERR_UNSUPPORTED  # K > 4
    assert bd.rssm_kda_spec_verify(st8.desc, 0, *args8) == bd.RSSM_ERR_INVALID_ARG
    assert bd.rssm_kda_spec_verify(st8.desc, 9, *args8) == bd.RSSM_ERR_INVALID_ARG  # K > L


def test_kda_verify_over_pending_is_reported():
    """A second verify before the commit is reported and changes nothing."""
    w = KW("kpend", 2, 2, 128, 128, 8, 1, seed=426, drafts=1, prefill=False)
    st, _, _, _ = kda_from_workload(w, "cuda")
    o = st.new_verify_output(w.n_new)
    rec = I.kda_verify_inputs(w, 0, "cuda")
    st.verify(rec, o)
    torch.cuda.synchronize()
    before = (st.S.clone(), st.cursors.clone(), st.re.clone(), st.rk.clone())
    st.verify(rec, o)
    torch.cuda.synchronize()
    assert H.status(st) == bd.RSSM_DEV_PENDING
    for x, y in zip(before, (st.S, st.cursors, st.re, st.rk)):
        assert torch.equal(x, y)
