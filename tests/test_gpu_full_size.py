"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (bf16 outputs), on sampled sequences the oracle replays one by one,
plus properties checked over the whole batch (cursor trace bit-exact against
the cursor model, outputs finite, untouched checkpoints bit-identical)."""
import numpy as np
import pytest
import torch

import harness as H
from oracle import cursors as oc
from oracle import sessions
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL_Y32, TOL_CKPT, TOL_BF16_EXCESS, TOL_READ_COPY = 1e-4, 1e-5, 2e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def spread(counts, n=4):
    """n sequence indices spanning the range of initial window counts."""
    order = np.argsort(counts.cpu().numpy(), kind="stable")
    idx = np.linspace(0, len(order) - 1, n).round().astype(int)
    return sorted(set(int(order[i]) for i in idx))


def test_mamba2_serving_full_size():
    """Batch 256, 128 heads, 64x128 state, 8 groups, L=16, staggered windows, 256 steps."""
    w = I.WORKLOADS["mamba2_serving"]
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev, bd.RSSM_BF16)
    seqs = spread(counts)
    feed = H.Feed()
    sess = sessions.mamba2_ar_session(H.F64(st.ckpt[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                      counts[seqs].cpu().numpy(), feed, H.F64(A), H.F64(D), w.buf_len)
    model = [(int(s), int(c), 0, 0) for s, c in zip(starts.cpu(), counts.cpu())]
    y = st.new_output()
    flushes = 0
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, seqs)
        prev = st.ckpt[seqs].clone()
        st.step(rec, A, D, y)
        exp = next(sess)
        assert H.bf16_excess(H.F64(y[seqs]), exp["y"]) <= TOL_BF16_EXCESS, t
        assert torch.isfinite(y).all()
        model = [oc.ar_step(c, w.buf_len)[0] for c in model]
        np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array(model))
        for i, b in enumerate(seqs):
            if exp["flushed"][i]:
                flushes += 1
                assert H.rel_l2(H.F64(st.ckpt[b]), exp["state"][i]) <= TOL_CKPT, (t, b)
            else:
                assert torch.equal(st.ckpt[b], prev[i]), (t, b)  # non-flush steps write no state
    assert flushes == len(seqs) * (w.steps // w.buf_len)
    assert H.status(st) == 0


def test_mamba2_serving_fp32_outputs():
    """The same layer with fp32 outputs, 40 steps (2 flush rounds), 1e-4 rel-L2."""
    w = I.WORKLOADS["mamba2_serving"]
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev, bd.RSSM_F32)
    seqs = spread(counts, 3)
    feed = H.Feed()
    sess = sessions.mamba2_ar_session(H.F64(st.ckpt[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                      counts[seqs].cpu().numpy(), feed, H.F64(A), H.F64(D), w.buf_len)
    y = st.new_output()
    for t in range(40):
        rec = I.mamba2_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, seqs)
        st.step(rec, A, D, y)
        exp = next(sess)
        assert H.rel_l2(H.F64(y[seqs]), exp["y"]) <= TOL_Y32, t
    assert H.status(st) == 0


def test_mamba2_spec_full_size():
    """Batch 512, K = 4 records per verify, accepted ~U{0..3}, 128 verify steps, flush on overflow."""
    w = I.WORKLOADS["mamba2_spec"]
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev, bd.RSSM_BF16)
    seqs = spread(counts, 3)
    fv, fk = H.Feed(), H.Feed()
    sess = sessions.mamba2_spec_session(H.F64(st.ckpt[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                        counts[seqs].cpu().numpy(), fv, fk, H.F64(A), H.F64(D), w.buf_len)
    model = [(int(s), int(c), 0, 0) for s, c in zip(starts.cpu(), counts.cpu())]
    y = st.new_output(w.n_new)
    folds = 0
    for t in range(w.steps):
        rec = I.mamba2_verify_inputs(w, t, dev)
        kept = I.accepted_kept(w, t, dev)
        fv.rec = H.sub(rec, seqs)
        fk.rec = kept[seqs].cpu().numpy()
        st.verify(rec, A, D, y)
        model = [oc.verify(c, w.n_new, w.buf_len)[0] for c in model]
        np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array(model))
        st.commit(kept)
        kl = kept.cpu().tolist()
        model = [oc.commit(c, k, w.buf_len)[0] for c, k in zip(model, kl)]
        np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array(model))
        exp = next(sess)
        assert H.bf16_excess(H.F64(y[seqs]), exp["y"]) <= TOL_BF16_EXCESS, t
        assert torch.isfinite(y).all()
        for i, b in enumerate(seqs):
            if exp["folded"][i]:
                folds += 1
                assert H.rel_l2(H.F64(st.ckpt[b]), exp["committed_state"][i]) <= TOL_CKPT, (t, b)
    assert folds > 0
    assert H.status(st) == 0


def test_gdn_serving_full_size():
    """Batch 256, 32 heads, 128x128 state, L=16, staggered windows, 256 steps."""
    w = I.WORKLOADS["gdn_serving"]
    dev = "cuda"
    st, pre, starts, counts = H.gdn_setup(w, dev, bd.RSSM_BF16)
    seqs = spread(counts, 3)
    feed = H.Feed()
    sess = sessions.gdn_ar_session(H.F64(st.S[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                   counts[seqs].cpu().numpy(), feed, w.buf_len)
    o = st.new_output()
    flushes = 0
    for t in range(w.steps):
        rec = I.gdn_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, seqs)
        st.step(rec, o)
        exp = next(sess)
        assert H.bf16_excess(H.F64(o[seqs]), exp["o"]) <= TOL_BF16_EXCESS, t
        for i, b in enumerate(seqs):
            if exp["flushed"][i]:
                flushes += 1
                assert H.rel_l2(H.F64(st.S[b]), exp["state"][i]) <= TOL_CKPT, (t, b)
    assert torch.isfinite(o).all()
    assert flushes == len(seqs) * (w.steps // w.buf_len)
    assert H.status(st) == 0


def test_kda_serving_full_size():
    """Kimi Delta Attention at the bench's size: batch 256, 32 heads, 128x128
    state, L=16, staggered windows, 256 steps; the cursor trace of the whole
    batch against the cursor model."""
    from recurrent_state_decode_gb300.state import kda_from_workload
    w = I.WORKLOADS["kda_serving"]
    dev = "cuda"
    st, pre, starts, counts = kda_from_workload(w, dev, bd.RSSM_BF16)
    seqs = spread(counts, 3)
    feed = H.Feed()
    sess = sessions.kda_ar_session(H.F64(st.S[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                   counts[seqs].cpu().numpy(), feed, w.buf_len)
    cur = [(int(a), int(c), 0, 0) for a, c in zip(starts.tolist(), counts.tolist())]
    o = st.new_output()
    flushes = 0
    for t in range(w.steps):
        rec = I.kda_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, seqs)
        st.step(rec, o)
        exp = next(sess)
        assert H.bf16_excess(H.F64(o[seqs]), exp["o"]) <= TOL_BF16_EXCESS, t
        for i, b in enumerate(seqs):
            if exp["flushed"][i]:
                flushes += 1
                assert H.rel_l2(H.F64(st.S[b]), exp["state"][i]) <= TOL_CKPT, (t, b)
        cur = [oc.ar_step(c, w.buf_len)[0] for c in cur]
        if t % 64 == 63:
            np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array(cur))
    assert torch.isfinite(o).all()
    assert flushes == len(seqs) * (w.steps // w.buf_len)
    assert H.status(st) == 0


def test_gdn_spec_full_size():
    """Gated DeltaNet speculative decode: batch 512, 32 heads, 128x128 state,
    K = 4 records per verify, accepted ~U{0..3}, 128 verify steps, fold on overflow."""
    w = I.WORKLOADS["gdn_spec"]
    dev = "cuda"
    st, pre, starts, counts = H.gdn_setup(w, dev, bd.RSSM_BF16)
    seqs = spread(counts, 3)
    fv, fk = H.Feed(), H.Feed()
    sess = sessions.gdn_spec_session(H.F64(st.S[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                     counts[seqs].cpu().numpy(), fv, fk, w.buf_len)
    model = [(int(s), int(c), 0, 0) for s, c in zip(starts.cpu(), counts.cpu())]
    o = st.new_verify_output(w.n_new)
    folds = 0
    for t in range(w.steps):
        rec = I.gdn_verify_inputs(w, t, dev)
        kept = I.accepted_kept(w, t, dev)
        fv.rec = H.sub(rec, seqs)
        fk.rec = kept[seqs].cpu().numpy()
        st.verify(rec, o)
        model = [oc.verify(c, w.n_new, w.buf_len)[0] for c in model]
        np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array(model))
        st.commit(kept)
        model = [oc.commit(c, k, w.buf_len)[0] for c, k in zip(model, kept.cpu().tolist())]
        np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array(model))
        exp = next(sess)
        assert H.bf16_excess(H.F64(o[seqs]), exp["o"]) <= TOL_BF16_EXCESS, t
        assert torch.isfinite(o).all()
        for i, b in enumerate(seqs):
            if exp["folded"][i]:
                folds += 1
                assert H.rel_l2(H.F64(st.S[b]), exp["committed_state"][i]) <= TOL_CKPT, (t, b)
    assert folds > 0
    assert H.status(st) == 0


@pytest.mark.parametrize("name", ["mamba2_bf16_read", "mamba2_f16_read", "mamba2_f8_read"])
def test_read_copy_4096_steps(name):
    """fp32 recurrence checkpoint + bf16 (or fp16) read copy, 4096 steps: the
    output error stays within 1e-2 relative L2 and does not grow (rounding of
    the read copy never enters the recurrence)."""
    w = I.WORKLOADS[name]
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev, bd.RSSM_F32)
    assert st.ckpt_read is not None
    seqs = spread(counts, 2)
    feed = H.Feed()
    sess = sessions.mamba2_ar_session(H.F64(st.ckpt[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                      counts[seqs].cpu().numpy(), feed, H.F64(A), H.F64(D), w.buf_len)
    y = st.new_output()
    trace = []
    worst_ckpt = 0.0
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, seqs)
        st.step(rec, A, D, y)
        exp = next(sess)
        trace.append(H.rel_l2(H.F64(y[seqs]), exp["y"]))
        for i, b in enumerate(seqs):
            if exp["flushed"][i]:
                worst_ckpt = max(worst_ckpt, H.rel_l2(H.F64(st.ckpt[b]), exp["state"][i]))
    trace = np.array(trace)
    assert trace.max() <= (2.0 ** -4 if w.read_copy == "f8" else TOL_READ_COPY)  # e4m3 half-ulp for fp8
    assert trace[-512:].max() <= 1.25 * trace[:512].max()
    slope = np.polyfit(np.arange(len(trace)), trace, 1)[0]
    assert slope < 1e-7, slope
    assert worst_ckpt <= TOL_CKPT
    assert H.status(st) == 0
