"""Mamba-2 parity on the GPU, through the C ABI, against the fp64 oracle.

Tolerances: fp32 outputs <= 1e-4 relative L2 per step; the checkpoint of
every sequence that flushed <= 1e-5 relative L2; bf16 outputs: the error
beyond half a bf16 ulp of the reference <= 2e-3 x output RMS; cursors
bit-exact; bf16 read copy outputs <= 1e-2 relative L2.
"""
import numpy as np
import pytest
import torch

import harness as H
from oracle import readcopy as rc
from oracle import sessions
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.state import Mamba2State
from recurrent_state_decode_gb300.inputs import Mamba2Workload as W

pytestmark = pytest.mark.gpu

TOL_READ_F8 = 2.0 ** -4  # e4m3 half-ulp: the largest relative error of a checkpoint element read
TOL_Y32, TOL_CKPT, TOL_BF16_EXCESS, TOL_READ_COPY = 1e-4, 1e-5, 2e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def run_ar(w, out_dtype=bd.RSSM_F32, seqs=None, read_copy=None, steps=None, trace=None):
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev, out_dtype, read_copy)
    rc_f8 = read_copy == "f8"
    read_copy = st.ckpt_read is not None
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    feed = H.Feed()
    sess = sessions.mamba2_ar_session(H.F64(st.ckpt[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                      counts[seqs].cpu().numpy(), feed, H.F64(A), H.F64(D), w.buf_len)
    y = st.new_output()
    flushes = 0
    for t in range(w.steps if steps is None else steps):
        rec = I.mamba2_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, seqs)
        st.step(rec, A, D, y)
        exp = next(sess)
        yg = H.F64(y[seqs])
        if read_copy:
            err = H.rel_l2(yg, exp["y"])
            if trace is not None:
                trace.append(err)
            assert err <= (TOL_READ_F8 if rc_f8 else TOL_READ_COPY), (t, err)
        elif out_dtype == bd.RSSM_F32:
            err = H.rel_l2(yg, exp["y"])
            assert err <= TOL_Y32, (t, err)
        else:
            ex = H.bf16_excess(yg, exp["y"])
            assert ex <= TOL_BF16_EXCESS, (t, ex)
        np.testing.assert_array_equal(st.cursors[seqs].cpu().numpy(), exp["cursors"])
        for i, b in enumerate(seqs):
            if exp["flushed"][i]:
                flushes += 1
                e = H.rel_l2(H.F64(st.ckpt[b]), exp["state"][i])
                assert e <= TOL_CKPT, (t, b, e)
                if read_copy:  # the read copy is the oracle's rounding of the new checkpoint, bit for bit
                    H.assert_read_copy(st, b)
    assert H.status(st) == 0
    return flushes


def test_tiny_fp32():
    """Batch 4, 8 heads, 64x128 state, L=16, 64 steps from a zero checkpoint."""
    assert run_ar(I.WORKLOADS["mamba2_tiny"]) == 4 * 4


def test_tiny_bf16_out():
    run_ar(I.WORKLOADS["mamba2_tiny"], out_dtype=bd.RSSM_BF16)


SHAPES = [
    W("ragged", 3, 6, 24, 40, 3, 5, 23, seed=11),          # dims off every tile size, groups of 2 heads
    W("L1", 2, 4, 16, 32, 2, 1, 6, seed=12),                # every step is a flush (L=1 is conventional decoding)
    W("L2", 3, 4, 16, 32, 4, 2, 9, seed=13),
    W("L32", 3, 4, 64, 128, 2, 32, 70, seed=14),            # largest window: the warp scan spans 32 records
    W("wideN", 2, 2, 32, 256, 1, 4, 9, seed=15),           # two column chunks per lane
    W("multiblock", 2, 2, 256, 256, 2, 3, 7, seed=16),     # 8 row blocks per (sequence, head)
    W("tiny_dims", 2, 2, 8, 8, 1, 3, 7, seed=17),          # one 8-row group, one partial chunk
    W("odd_batch", 5, 3, 40, 72, 3, 7, 15, seed=18),
    W("fast_p192", 2, 4, 192, 128, 2, 8, 19, seed=25),    # shape-specialised kernel, three row blocks per head
    W("fast_L31", 2, 2, 64, 128, 1, 31, 40, seed=26),     # its longest window
    W("fast_hpg1", 3, 3, 64, 128, 3, 6, 14, seed=27),     # one head per group
]


@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
@pytest.mark.parametrize("out", [bd.RSSM_F32, bd.RSSM_BF16], ids=["f32", "bf16"])
def test_shapes(w, out):
    run_ar(w, out_dtype=out)


READ_COPY = [
    SHAPES[0], SHAPES[3],
    W("rc", 3, 4, 64, 128, 2, 16, 40, seed=19),            # two heads of a group per block
    W("rc_g1", 2, 3, 64, 128, 3, 8, 20, seed=20),          # one head per group: one head per block
    W("rc_p128", 2, 4, 128, 128, 2, 8, 20, seed=21),       # two row blocks per head
    W("rc_L31", 2, 4, 64, 128, 1, 31, 70, seed=22),        # longest window of the shape-specialised kernels
    W("rc_L1", 2, 4, 64, 128, 2, 1, 5, seed=23),           # every step flushes
    W("rc_hpg4", 2, 8, 64, 128, 2, 5, 12, seed=24),        # two head pairs per group
]


@pytest.mark.parametrize("w", READ_COPY, ids=lambda w: w.name)
@pytest.mark.parametrize("rc", [True, "f16"], ids=["bf16", "f16"])
def test_read_copy_small(w, rc):
    run_ar(w, read_copy=rc)


@pytest.mark.parametrize("w", READ_COPY[2:], ids=lambda w: w.name)  # the shape-specialised shapes
def test_read_copy_f8(w):
    run_ar(w, read_copy="f8")


def test_conventional_kernel():
    """The comparison kernel: state read + written every step."""
    w = W("conv", 3, 6, 24, 40, 3, 16, 20, seed=21)
    dev = "cuda"
    from oracle import mamba2 as om
    A, D = I.mamba2_params(w, dev)
    state = I.mamba2_checkpoint(w, dev)
    h = H.F64(state)
    y = torch.empty((w.batch, w.nheads, w.headdim), device=dev)
    desc = bd.mamba2_desc(w.batch, w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len)
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, dev)
        bd.check(bd.rssm_mamba2_conventional_step(desc, state, rec["x"], rec["z"], rec["B"], rec["C"], rec["dt"],
                                                  A, D, y))
        r = {k: H.F64(v) for k, v in rec.items()}
        h, ye = om.conventional_step_layer(h, r["x"], r["z"], r["B"], r["C"], r["dt"], H.F64(A), H.F64(D))
        assert H.rel_l2(H.F64(y), ye) <= TOL_Y32
        assert H.rel_l2(H.F64(state), h) <= TOL_CKPT


def test_standalone_flush():
    """After some AR steps, a flush folds every non-empty window into the checkpoint."""
    w = W("flush", 4, 4, 32, 64, 2, 8, 5, seed=31)
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev)
    feed = H.Feed()
    sess = sessions.mamba2_ar_session(H.F64(st.ckpt), H.sub(pre, slice(None)), starts.cpu().numpy(),
                                      counts.cpu().numpy(), feed, H.F64(A), H.F64(D), w.buf_len)
    y = st.new_output()
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, dev)
        feed.rec = H.sub(rec, slice(None))
        st.step(rec, A, D, y)
        exp = next(sess)
    before = st.cursors.clone()
    st.flush(A)
    cur = st.cursors.cpu().numpy()
    bc = before.cpu().numpy()
    np.testing.assert_array_equal(cur[:, 0], (bc[:, 0] + bc[:, 1]) % w.buf_len)
    np.testing.assert_array_equal(cur[:, 1:], 0)
    for b in range(w.batch):
        assert H.rel_l2(H.F64(st.ckpt[b]), exp["state"][b]) <= TOL_CKPT
    # decoding continues correctly from the folded checkpoint
    rec = I.mamba2_step_inputs(w, 99, dev)
    feed.rec = H.sub(rec, slice(None))
    st.step(rec, A, D, y)
    exp = next(sess)
    assert H.rel_l2(H.F64(y), exp["y"]) <= TOL_Y32
    assert H.status(st) == 0


def run_spec(w, seqs=None, steps=None, out_dtype=bd.RSSM_F32, read_copy=None):
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev, out_dtype, read_copy)
    rc_f8 = read_copy == "f8"
    read_copy = st.ckpt_read is not None
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    fv, fk = H.Feed(), H.Feed()
    sess = sessions.mamba2_spec_session(H.F64(st.ckpt[seqs]), H.sub(pre, seqs), starts[seqs].cpu().numpy(),
                                        counts[seqs].cpu().numpy(), fv, fk, H.F64(A), H.F64(D), w.buf_len)
    y = st.new_output(w.n_new)
    folds = 0
    for t in range(w.steps if steps is None else steps):
        rec = I.mamba2_verify_inputs(w, t, dev)
        kept = I.accepted_kept(w, t, dev)
        fv.rec = H.sub(rec, seqs)
        fk.rec = kept[seqs].cpu().numpy()
        st.verify(rec, A, D, y)
        cv = st.cursors[seqs].cpu().numpy()
        st.commit(kept)
        exp = next(sess)
        yg = H.F64(y[seqs])
        if read_copy:
            assert H.rel_l2(yg, exp["y"]) <= (TOL_READ_F8 if rc_f8 else TOL_READ_COPY), t
        elif out_dtype == bd.RSSM_F32:
            assert H.rel_l2(yg, exp["y"]) <= TOL_Y32, t
        else:
            assert H.bf16_excess(yg, exp["y"]) <= TOL_BF16_EXCESS, t
        np.testing.assert_array_equal(cv, exp["cursors_verify"])
        np.testing.assert_array_equal(st.cursors[seqs].cpu().numpy(), exp["cursors_commit"])
        for i, b in enumerate(seqs):
            if exp["folded"][i]:
                folds += 1
                assert H.rel_l2(H.F64(st.ckpt[b]), exp["committed_state"][i]) <= TOL_CKPT, (t, b)
    assert H.status(st) == 0
    return folds


SPEC = [
    W("spec_small", 4, 4, 32, 64, 2, 16, 20, seed=41, drafts=3),
    W("spec_ragged", 3, 6, 24, 40, 3, 5, 12, seed=42, drafts=2),
    W("spec_K_eq_L", 3, 2, 16, 32, 1, 4, 8, seed=43, drafts=3),    # K = L: every verify with count > 0 folds
    W("spec_K1", 3, 2, 16, 32, 1, 4, 10, seed=44, drafts=0),       # single record per verify
    W("spec_fast_p128", 2, 4, 128, 128, 2, 8, 12, seed=46, drafts=3),   # shape-specialised verify, two row blocks
    W("spec_fast_L31_K1", 2, 2, 64, 128, 1, 31, 40, seed=47, drafts=0),  # L + K = 32, the longest view
    W("spec_fast_L28", 2, 2, 64, 128, 2, 28, 30, seed=48, drafts=3),     # L + K = 32 with four records
]


@pytest.mark.parametrize("w", SPEC, ids=lambda w: w.name)
def test_spec(w):
    assert run_spec(w) > 0 or w.name in ("spec_K1", "spec_fast_L31_K1")


def test_spec_bf16_out_and_read_copy():
    run_spec(SPEC[0], out_dtype=bd.RSSM_BF16)
    run_spec(SPEC[0], read_copy=True)
    run_spec(SPEC[0], read_copy="f16")
    run_spec(W("spec_fast", 3, 4, 64, 128, 2, 16, 12, seed=45, drafts=3), read_copy="f16")
    run_spec(W("spec_fast", 3, 4, 64, 128, 2, 16, 12, seed=45, drafts=3), read_copy="f8")


def test_spec_all_accepted_equals_ar():
    """With every draft kept, speculative decode must produce AR decode's outputs
    and checkpoint for the same token sequence (compared GPU to GPU)."""
    w = W("acc", 2, 4, 32, 64, 2, 16, 6, seed=51, drafts=3, prefill=False)
    dev = "cuda"
    sa, A, D, _, _, _ = H.mamba2_setup(w, dev)
    ss, _, _, _, _, _ = H.mamba2_setup(w, dev)
    ya = sa.new_output()
    ys = ss.new_output(w.n_new)
    kept = torch.full((w.batch,), w.n_new, dtype=torch.int32, device=dev)
    for t in range(w.steps):
        rec = I.mamba2_verify_inputs(w, t, dev)
        ss.verify(rec, A, D, ys)
        ss.commit(kept)
        for i in range(w.n_new):
            sa.step({k: v[:, i].contiguous() for k, v in rec.items()}, A, D, ya)
            assert H.rel_l2(H.F64(ys[:, i]), H.F64(ya)) <= TOL_Y32
    # flush both and compare checkpoints
    sa.flush(A)
    ss.flush(A)
    assert H.rel_l2(H.F64(ss.ckpt), H.F64(sa.ckpt)) <= TOL_CKPT
    assert H.status(sa) == 0 and H.status(ss) == 0


# ----------------------------------------------------------------------------- device-side errors

@pytest.mark.parametrize("w", [W("err", 4, 2, 16, 32, 1, 4, 1, seed=61, prefill=False),
                               W("err_fast", 4, 2, 64, 128, 1, 4, 1, seed=61, prefill=False)],
                         ids=lambda w: w.name)  # generic kernel + cursor kernel; fused cursor advance
def test_device_errors_skip_sequence(w):
    dev = "cuda"
    st, A, D, _, _, _ = H.mamba2_setup(w, dev)
    st.cursors[1] = torch.tensor([0, 7, 0, 0], dtype=torch.int32)     # count > L
    st.cursors[2] = torch.tensor([0, 1, 2, 0], dtype=torch.int32)     # uncommitted drafts
    st.cursors[3] = torch.tensor([0, 4, 0, 0], dtype=torch.int32)     # full window
    before = st.cursors.clone()
    ck = st.ckpt.clone()
    y = st.new_output().fill_(float("nan"))
    st.step(I.mamba2_step_inputs(w, 0, dev), A, D, y)
    torch.cuda.synchronize()
    assert H.status(st) == bd.RSSM_DEV_BAD_CURSOR or H.status(st) in (bd.RSSM_DEV_PENDING, bd.RSSM_DEV_WINDOW_FULL)
    assert torch.isfinite(y[0]).all()
    assert torch.isnan(y[1:]).all()
    assert torch.equal(st.cursors[1:], before[1:])
    assert torch.equal(st.ckpt, ck)
    assert st.cursors[0, 1].item() == 1


def test_commit_and_reset_errors():
    dev = "cuda"
    cur = torch.tensor([[0, 2, 3, 0], [1, 1, 2, 1], [0, 0, 0, 0]], dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kept = torch.tensor([4, 2, 0], dtype=torch.int32, device=dev)   # seq 0: kept > pending
    bd.check(bd.rssm_commit_cursors(cur, kept, 3, 4, status))
    torch.cuda.synchronize()
    assert status.item() == bd.RSSM_DEV_BAD_KEPT
    assert cur.cpu().tolist() == [[0, 2, 3, 0], [2, 2, 0, 0], [0, 0, 0, 0]]   # seq 1 folded: start 1+1, count 0+2
    status.zero_()
    slots = torch.tensor([1, 5], dtype=torch.int32, device=dev)
    bd.check(bd.rssm_reset_cursors(cur, slots, 2, 3, status))
    torch.cuda.synchronize()
    assert status.item() == bd.RSSM_DEV_BAD_SLOT
    assert cur.cpu().tolist() == [[0, 2, 3, 0], [0, 0, 0, 0], [0, 0, 0, 0]]


@pytest.mark.parametrize("w", [W("twice", 2, 2, 16, 32, 1, 8, 1, seed=62, drafts=1, prefill=False),
                               W("twice_fast", 2, 2, 64, 128, 1, 8, 1, seed=62, drafts=1, prefill=False)],
                         ids=lambda w: w.name)
def test_verify_twice_is_rejected(w):
    dev = "cuda"
    st, A, D, _, _, _ = H.mamba2_setup(w, dev)
    y = st.new_output(w.n_new)
    rec = I.mamba2_verify_inputs(w, 0, dev)
    st.verify(rec, A, D, y)
    st.verify(rec, A, D, y)
    torch.cuda.synchronize()
    assert H.status(st) == bd.RSSM_DEV_PENDING
    assert st.cursors[:, 2].tolist() == [2, 2]
    assert st.cursors[:, 3].tolist() == [0, 0]  # flags (and the arrival count) untouched by the rejected call


def test_downcast_rne():
    dev = "cuda"
    x = torch.randn(1001, device=dev) * 3
    x[:5] = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, float("inf"), 1e-40])  # ties to even, signed zero, inf, subnormal
    out = torch.empty(1001, dtype=torch.bfloat16, device=dev)
    bd.check(bd.rssm_checkpoint_downcast(x, out, 1001, bd.RSSM_BF16))
    xs = x.cpu().numpy()
    np.testing.assert_array_equal(H.bits16(out), rc.bf16_bits(rc.to_bf16(xs)))
    # fp16: ties to even at 1 + 2^-11 and 1 + 3 * 2^-11, overflow to inf, fp16 subnormals
    x[:5] = torch.tensor([1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 70000.0, -3e-6, 2 ** -25])
    h = torch.empty(1001, dtype=torch.float16, device=dev)
    bd.check(bd.rssm_checkpoint_downcast(x, h, 1001, bd.RSSM_F16))
    xs = x.cpu().numpy()
    np.testing.assert_array_equal(H.bits16(h), rc.fp16_bits(rc.to_fp16(xs)))


def test_downcast_f8_rows():
    """The fp8 read copy of a whole checkpoint: e4m3 bytes and row scales equal
    the scaled round-to-nearest-even conversion, row by row (zero rows, rows
    whose max is negative, a row of one value)."""
    w = W("f8dc", 3, 2, 64, 128, 1, 8, 1, seed=64)
    st = Mamba2State(w.batch, w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len, "cuda", read_copy="f8")
    st.ckpt.copy_(torch.randn_like(st.ckpt) * torch.logspace(-6, 3, 128, device="cuda"))
    st.ckpt[0, 0, 0] = 0.0
    st.ckpt[0, 0, 1] = -torch.rand(128, device="cuda") - 1.0
    st.ckpt[0, 1, 2] = 3.25
    st.downcast()
    q, sc = rc.e4m3_rows(st.ckpt.cpu().numpy())
    np.testing.assert_array_equal(st.read_q.cpu().numpy(), q)
    np.testing.assert_array_equal(st.read_scale.cpu().numpy(), sc)
    assert st.read_scale[0, 0, 0].item() == 0.0


def test_reset_then_decode():
    """A reset slot restarts from its (caller-written) checkpoint with an empty window."""
    w = W("reset", 3, 2, 16, 32, 1, 4, 6, seed=63)
    dev = "cuda"
    st, A, D, pre, starts, counts = H.mamba2_setup(w, dev)
    y = st.new_output()
    for t in range(3):
        st.step(I.mamba2_step_inputs(w, t, dev), A, D, y)
    st.ckpt[1].zero_()
    st.reset(torch.tensor([1], dtype=torch.int32, device=dev))
    assert st.cursors[1].tolist() == [0, 0, 0, 0]
    from oracle import mamba2 as om
    h = np.zeros((1, w.nheads, w.headdim, w.dstate))
    for t in range(3, 3 + w.steps):
        rec = I.mamba2_step_inputs(w, t, dev)
        st.step(rec, A, D, y)
        r = {k: H.F64(v[1:2]) for k, v in rec.items()}
        h, ye = om.conventional_step_layer(h, r["x"], r["z"], r["B"], r["C"], r["dt"], H.F64(A), H.F64(D))
        assert H.rel_l2(H.F64(y[1:2]), ye) <= TOL_Y32
    assert H.status(st) == 0
