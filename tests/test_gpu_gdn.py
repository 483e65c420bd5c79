"""Gated DeltaNet parity on the GPU, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import harness as H
from oracle import gdn as og
from oracle import sessions
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import GDNWorkload as GW

pytestmark = pytest.mark.gpu

TOL_Y32, TOL_CKPT, TOL_BF16_EXCESS = 1e-4, 1e-5, 2e-3


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def run_gdn(w, out_dtype=bd.RSSM_F32, seqs=None, steps=None):
    dev = "cuda"
    st, pre, starts, counts = H.gdn_setup(w, dev, out_dtype)
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    feed = H.Feed()
    sess = sessions.gdn_ar_session(H.F64(st.S[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                   counts[seqs].cpu().numpy(), feed, w.buf_len)
    o = st.new_output()
    flushes = 0
    for t in range(w.steps if steps is None else steps):
        rec = I.gdn_step_inputs(w, t, dev)
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


GSHAPES = [
    GW("gdn_small", 3, 2, 64, 64, 16, 40, seed=71),
    GW("gdn_ragged", 3, 3, 40, 24, 5, 17, seed=72),          # dk, dv off the chunk sizes
    GW("gdn_L1", 2, 2, 32, 32, 1, 5, seed=73),
    GW("gdn_L32", 2, 2, 32, 48, 32, 70, seed=74),
    GW("gdn_big_tile", 2, 1, 256, 256, 4, 9, seed=75),       # 4 row blocks, 16 chunks per thread
    GW("gdn_128", 2, 4, 128, 128, 16, 34, seed=76),          # the serving tile (shape-specialised kernel)
    GW("gdn_128_L1", 2, 3, 128, 128, 1, 6, seed=79),         # every step flushes
    GW("gdn_128_L5", 3, 2, 128, 128, 5, 23, seed=80),        # ragged window, wraps often
    GW("gdn_128_L31", 2, 2, 128, 128, 31, 70, seed=81),      # longest window of that kernel
    GW("gdn_128_H3", 3, 3, 128, 128, 7, 20, seed=85),         # odd head count
]


@pytest.mark.parametrize("w", GSHAPES, ids=lambda w: w.name)
@pytest.mark.parametrize("out", [bd.RSSM_F32, bd.RSSM_BF16], ids=["f32", "bf16"])
def test_gdn_shapes(w, out):
    run_gdn(w, out)


def test_gdn_conventional_kernel():
    w = GW("gconv", 3, 3, 40, 24, 16, 20, seed=77)
    dev = "cuda"
    S = I.gdn_checkpoint(w, dev)
    Sh = H.F64(S)
    o = torch.empty((w.batch, w.nheads, w.dv), device=dev)
    desc = bd.gdn_desc(w.batch, w.nheads, w.dk, w.dv, w.buf_len)
    for t in range(w.steps):
        rec = I.gdn_step_inputs(w, t, dev)
        bd.check(bd.rssm_gdn_conventional_step(desc, S, rec["q"], rec["k"], rec["v"], rec["g"], rec["beta"], o))
        r = {k: H.F64(v) for k, v in rec.items()}
        Sh, oe = og.conventional_step(Sh, r["q"], r["k"], r["v"], r["g"], r["beta"])
        assert H.rel_l2(H.F64(o), oe) <= TOL_Y32
        assert H.rel_l2(H.F64(S), Sh) <= TOL_CKPT


def test_gdn_standalone_flush():
    w = GW("gflush", 3, 2, 32, 40, 8, 5, seed=78)
    dev = "cuda"
    st, pre, starts, counts = H.gdn_setup(w, dev)
    feed = H.Feed()
    sess = sessions.gdn_ar_session(H.F64(st.S), H.sub(pre, slice(None)), starts.cpu().numpy(), counts.cpu().numpy(),
                                   feed, w.buf_len)
    o = st.new_output()
    for t in range(w.steps):
        rec = I.gdn_step_inputs(w, t, dev)
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


@pytest.mark.parametrize("w", [GW("gprime", 3, 2, 128, 128, 16, 1, seed=82),
                               GW("gprime_small", 3, 2, 40, 24, 7, 1, seed=83)], ids=lambda w: w.name)
def test_gdn_prime_matches_window_corrections(w):
    """rssm_gdn_prime fills ring.e with each window record's correction e_t,
    checked against the oracle's forward substitution."""
    st, pre, starts, counts = H.gdn_setup(w, "cuda")  # places the windows, then primes
    S0 = H.F64(st.S)
    re = H.F64(st.re)
    checked = 0
    for b in range(w.batch):
        c, s0 = int(counts[b]), int(starts[b])
        if c == 0:
            continue
        r = {k: H.F64(v[b, :c]) for k, v in pre.items()}  # [c, H, ...]
        ks, vs = np.moveaxis(r["k"], 0, 1), np.moveaxis(r["v"], 0, 1)
        gs, bs = r["g"].T, r["beta"].T
        _, e = og._window_terms(S0[b], ks, vs, gs, bs)  # e [H, c, dv]
        slots = [(s0 + t) % w.buf_len for t in range(c)]
        assert H.rel_l2(re[b][:, slots], e) <= 1e-5
        checked += 1
    assert checked > 0
    assert H.status(st) == 0


@pytest.mark.parametrize("w", [GW("gerr", 3, 2, 40, 24, 4, 1, seed=84, prefill=False),
                               GW("gerr_fast", 3, 2, 128, 128, 4, 1, seed=84, prefill=False)],
                         ids=lambda w: w.name)
def test_gdn_device_errors_skip_sequence(w):
    """Bad cursors are reported, left as they were and skipped; the other sequences step."""
    dev = "cuda"
    st, _, _, _ = H.gdn_setup(w, dev)
    st.cursors[1] = torch.tensor([0, 7, 0, 0], dtype=torch.int32)  # count > L
    st.cursors[2] = torch.tensor([0, 1, 2, 0], dtype=torch.int32)  # uncommitted drafts
    before = st.cursors.clone()
    S0 = st.S.clone()
    o = st.new_output().fill_(float("nan"))
    st.step(I.gdn_step_inputs(w, 0, dev), o)
    torch.cuda.synchronize()
    assert H.status(st) in (bd.RSSM_DEV_BAD_CURSOR, bd.RSSM_DEV_PENDING)
    assert torch.isfinite(o[0]).all()
    assert torch.isnan(o[1:]).all()
    assert torch.equal(st.cursors[1:], before[1:])
    assert st.cursors[0].tolist() == [0, 1, 0, 0]
    assert torch.equal(st.S[1:], S0[1:])


# ----------------------------------------------------------------------------- speculative verify

def run_gdn_spec(w, out_dtype=bd.RSSM_F32, seqs=None, steps=None):
    dev = "cuda"
    st, pre, starts, counts = H.gdn_setup(w, dev, out_dtype)
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    fv, fk = H.Feed(), H.Feed()
    sess = sessions.gdn_spec_session(H.F64(st.S[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                     counts[seqs].cpu().numpy(), fv, fk, w.buf_len)
    o = st.new_verify_output(w.n_new)
    folds = 0
    for t in range(w.steps if steps is None else steps):
        rec = I.gdn_verify_inputs(w, t, dev)
        kept = I.accepted_kept(w, t, dev)
        fv.rec = H.sub(rec, seqs)
        fk.rec = kept[seqs].cpu().numpy()
        st.verify(rec, o)
        cv = st.cursors[seqs].cpu().numpy()
        st.commit(kept)
        exp = next(sess)
        og_ = H.F64(o[seqs])
        if out_dtype == bd.RSSM_F32:
            assert H.rel_l2(og_, exp["o"]) <= TOL_Y32, t
        else:
            assert H.bf16_excess(og_, exp["o"]) <= TOL_BF16_EXCESS, t
        np.testing.assert_array_equal(cv, exp["cursors_verify"])
        np.testing.assert_array_equal(st.cursors[seqs].cpu().numpy(), exp["cursors_commit"])
        for i, b in enumerate(seqs):
            if exp["folded"][i]:
                folds += 1
                assert H.rel_l2(H.F64(st.S[b]), exp["committed_state"][i]) <= TOL_CKPT, (t, b)
    assert H.status(st) == 0
    return folds


GSPEC = [
    GW("gspec_small", 3, 2, 64, 64, 16, 20, seed=91, drafts=3),
    GW("gspec_ragged", 3, 3, 40, 24, 5, 12, seed=92, drafts=2),
    GW("gspec_K_eq_L", 3, 2, 32, 32, 4, 8, seed=93, drafts=3),      # K = L: every verify with count > 0 folds
    GW("gspec_K1", 3, 2, 32, 48, 4, 10, seed=94, drafts=0),         # one record per verify
    GW("gspec_128", 3, 4, 128, 128, 16, 24, seed=95, drafts=3),     # the serving tile
    GW("gspec_128_L5", 2, 2, 128, 128, 5, 14, seed=96, drafts=3),   # folds often
    GW("gspec_128_K1", 2, 2, 128, 128, 8, 12, seed=98, drafts=0),
    GW("gspec_128_K2", 3, 2, 128, 128, 8, 12, seed=99, drafts=1),
    GW("gspec_128_L28", 2, 2, 128, 128, 28, 24, seed=100, drafts=3),  # L + K = 32, the longest view
]


@pytest.mark.parametrize("w", GSPEC, ids=lambda w: w.name)
def test_gdn_spec(w):
    assert run_gdn_spec(w) > 0 or w.name in ("gspec_K1", "gspec_128_K1")


def test_gdn_spec_bf16_out():
    run_gdn_spec(GSPEC[4], out_dtype=bd.RSSM_BF16)


def test_gdn_spec_all_accepted_equals_ar():
    """Every draft kept: speculative decode produces AR decode's outputs and
    state for the same tokens (GPU against GPU, then a flush of both)."""
    w = GW("gacc", 2, 2, 128, 128, 16, 6, seed=97, drafts=3, prefill=False)
    dev = "cuda"
    sa, _, _, _ = H.gdn_setup(w, dev)
    ss, _, _, _ = H.gdn_setup(w, dev)
    oa = sa.new_output()
    os_ = ss.new_verify_output(w.n_new)
    for t in range(w.steps):
        rec = I.gdn_verify_inputs(w, t, dev)
        ss.verify(rec, os_)
        ss.commit(torch.full((w.batch,), w.n_new, dtype=torch.int32, device=dev))
        for i in range(w.n_new):
            sa.step({k: v[:, i].contiguous() for k, v in rec.items()}, oa)
            assert H.rel_l2(H.F64(os_[:, i]), H.F64(oa)) <= TOL_Y32, (t, i)
    sa.flush()
    ss.flush()
    assert H.rel_l2(H.F64(ss.S), H.F64(sa.S)) <= TOL_CKPT
    assert H.status(sa) == 0 and H.status(ss) == 0


@pytest.mark.parametrize("w", [GW("gtwice", 2, 2, 40, 24, 8, 1, seed=101, drafts=1, prefill=False),
                               GW("gtwice_fast", 2, 2, 128, 128, 8, 1, seed=101, drafts=1, prefill=False)],
                         ids=lambda w: w.name)
def test_gdn_verify_twice_is_rejected(w):
    dev = "cuda"
    st, _, _, _ = H.gdn_setup(w, dev)
    o = st.new_verify_output(w.n_new)
    rec = I.gdn_verify_inputs(w, 0, dev)
    st.verify(rec, o)
    st.verify(rec, o)
    torch.cuda.synchronize()
    assert H.status(st) == bd.RSSM_DEV_PENDING
    assert st.cursors.cpu().tolist() == [[0, 0, 2, 0], [0, 0, 2, 0]]
