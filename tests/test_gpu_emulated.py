"""Emulated read precisions (rssm_mamba2_step_emulated) against the oracle.

A non-flush step reads the fp32 checkpoint through a quantise-dequantise in
the chosen format; a flushing step reads and folds the exact checkpoint
("ReplaySSM", the paper's code repository, introduction: the emulation
kernels implement separate read and recurrence precision and expose their
quantization behavior). The oracle's emulate_read of the GPU's own fp32
checkpoint gives the values a step reads (the codes are decided in fp32 on
both sides, so the reads agree exactly); its replay formula over the window
gives the expected output (fp32 path: <= 1e-4 relative L2); its
emulation_error gives the expected error report (<= 1e-5 relative). Flushed
checkpoints are checked against the conventional session (<= 1e-5).
The emulated reads are also checked, bit for bit, against the stored read
copies: the emulated bf16 read against the stored bf16 copy, and the
emulated e4m3 read with a row scale against the stored fp8 copy (the two
paths scale, convert and read back separately).
"""
import numpy as np
import pytest
import torch

import harness as H
from oracle import mamba2 as om
from oracle import readcopy as rc
from oracle import sessions
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import Mamba2Workload as W
from recurrent_state_decode_gb300.state import mamba2_from_workload

pytestmark = pytest.mark.gpu

TOL_Y32, TOL_CKPT, TOL_ERR = 1e-4, 1e-5, 1e-5
DEV = "cuda"
FMT = {"bf16": bd.RSSM_EMU_BF16, "fp16": bd.RSSM_EMU_F16, "e4m3": bd.RSSM_EMU_E4M3, "e5m2": bd.RSSM_EMU_E5M2,
       "int8": bd.RSSM_EMU_INT8}
SCALE = {"none": bd.RSSM_EMU_SCALE_NONE, "row": bd.RSSM_EMU_SCALE_ROW, "tile64": bd.RSSM_EMU_SCALE_TILE64}
PAIRS = [("bf16", "none"), ("fp16", "none"), ("e4m3", "row"), ("e4m3", "tile64"), ("e5m2", "row"),
         ("int8", "row"), ("int8", "tile64")]


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def emu_buffers(st):
    n = bd.rssm_mamba2_emulated_workspace_bytes(st.desc)
    return torch.zeros(2, dtype=torch.float64, device=DEV), torch.empty(n, dtype=torch.uint8, device=DEV)


def window_of(st, b, w):
    """Sequence b's window records from the GPU ring (cursor order): x [m,H,P],
    B [m,G,N], dt [m,H] as fp64."""
    start, count = (int(v) for v in st.cursors[b, :2].tolist())
    slots = [(start + j) % w.buf_len for j in range(count)]
    return (H.F64(st.rx[b][:, slots].transpose(0, 1)), H.F64(st.rB[b][:, slots].transpose(0, 1)),
            H.F64(st.rdt[b][:, slots].transpose(0, 1)))


def expected_outputs(st, rec, A, D, w, fmt, scale):
    """The oracle's output of every sequence for this step, reading the
    checkpoint through emulate_read on non-flush steps and exactly on a
    flushing one, and the error report's (sum of squared errors, sum of squares)."""
    y = np.zeros((w.batch, w.nheads, w.headdim))
    e_sum = n_sum = 0.0
    G = om.group_of_head(w.nheads, w.ngroups)
    A64, D64 = H.F64(A), H.F64(D)
    for b in range(w.batch):
        h0 = st.ckpt[b].cpu().numpy()
        xs, Bs, dts = window_of(st, b, w)
        flush = xs.shape[0] + 1 == w.buf_len
        if flush:
            hread = h0.astype(np.float64)
        else:
            hread = rc.emulate_read(h0, fmt, scale)
            e, n = rc.emulation_error(h0, fmt, scale)
            e_sum, n_sum = e_sum + e, n_sum + n
        x, z = H.F64(rec["x"][b]), H.F64(rec["z"][b])
        Bc, Cc, dt = H.F64(rec["B"][b]), H.F64(rec["C"][b]), H.F64(rec["dt"][b])
        xs_all = np.concatenate([xs, x[None]], 0).transpose(1, 0, 2)          # [H, m, P]
        Bs_all = np.concatenate([Bs[:, G], Bc[None, G]], 0).transpose(1, 0, 2)  # [H, m, N]
        dts_all = np.concatenate([dts, dt[None]], 0).T                        # [H, m]
        y[b] = om.replay_output(hread, xs_all, Bs_all, dts_all, Cc[G], z, A64, D64)
    return y, e_sum, n_sum


@pytest.mark.parametrize("fmt,scale", PAIRS, ids=[f"{f}-{s}" for f, s in PAIRS])
def test_emulated_step_against_the_oracle(fmt, scale):
    # headdim 128: two 64-row tiles per head (the tile scale is per 64-row block);
    # L = 6 and 14 steps: flushes on the way, from staggered windows
    w = W("emu", 3, 4, 128, 128, 2, 6, 14, seed=601)
    st, A, D, pre, starts, counts = mamba2_from_workload(w, DEV, bd.RSSM_F32, read_copy=False)
    err, ws = emu_buffers(st)
    emu = bd.emulation(FMT[fmt], SCALE[scale])
    feed = H.Feed()
    sess = sessions.mamba2_ar_session(H.F64(st.ckpt), H.sub(pre, slice(None)), starts.cpu().numpy(),
                                      counts.cpu().numpy(), feed, H.F64(A), H.F64(D), w.buf_len)
    y = st.new_output()
    flushes = 0
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, DEV)
        feed.rec = H.sub(rec, slice(None))
        y_exp, e_exp, n_exp = expected_outputs(st, rec, A, D, w, fmt, scale)
        st.step_emulated(rec, A, D, y, emu, err, ws)
        exp = next(sess)
        assert H.rel_l2(H.F64(y), y_exp) <= TOL_Y32, t
        e_gpu, n_gpu = err.tolist()
        assert n_gpu == pytest.approx(n_exp, rel=TOL_ERR), t
        assert e_gpu == pytest.approx(e_exp, rel=TOL_ERR, abs=1e-30), t
        np.testing.assert_array_equal(st.cursors.cpu().numpy(), exp["cursors"])
        for b in np.nonzero(exp["flushed"])[0]:
            flushes += 1
            assert H.rel_l2(H.F64(st.ckpt[b]), exp["state"][b]) <= TOL_CKPT, (t, b)
    assert flushes >= w.batch
    assert H.status(st) == 0


@pytest.mark.parametrize("fmt,read_copy", [("bf16", True), ("e4m3", "f8")])
def test_emulated_read_equals_the_stored_read_copy(fmt, read_copy):
    """The emulated bf16 read (no scale) and e4m3 read (row scale) are the
    stored bf16 and fp8 read copies of the same checkpoint: the emulated
    path's scaling and conversion against the stored copies', bit for bit,
    through the outputs."""
    w = W("emu_rc", 3, 8, 64, 128, 2, 8, 12, seed=602)
    se, A, D, _, _, _ = mamba2_from_workload(w, DEV, bd.RSSM_F32, read_copy=False)
    sr, _, _, _, _, _ = mamba2_from_workload(w, DEV, bd.RSSM_F32, read_copy=read_copy)
    err, ws = emu_buffers(se)
    emu = bd.emulation(FMT[fmt], SCALE["none" if fmt == "bf16" else "row"])
    ye, yr = se.new_output(), sr.new_output()
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, DEV)
        se.step_emulated(rec, A, D, ye, emu, err, ws)
        sr.step(rec, A, D, yr)
        torch.cuda.synchronize()
        assert torch.equal(ye, yr), t
    assert torch.equal(se.ckpt, sr.ckpt)
    assert H.status(se) == 0 and H.status(sr) == 0


def test_emulated_quantiser_against_the_oracle_rounding():
    """A checkpoint of values chosen to hit every rounding case (ties, the
    format-subnormal ranges, saturation): a one-step emulated read of it
    (no window, so y = h . C with C a unit vector picks one column) equals
    the oracle's rounding, element by element, for every format."""
    w = W("emu_q", 1, 1, 64, 128, 1, 4, 1, seed=603, prefill=False, zero_ckpt=True)
    g = np.random.default_rng(604)
    vals = np.concatenate([
        g.standard_normal(4096) * 10.0 ** g.uniform(-9, 2, 4096),
        (1 + np.arange(0, 64) / 64.0) * 2.0 ** g.integers(-30, 10, 64),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -11, 2.0 ** -14, 2.0 ** -25, 2.0 ** -10, 3 * 2.0 ** -11,
                  448.0, 460.0, 500.0, 57344.0, 6e4, 1e5, -0.0, 2.0 ** -126, 2.0 ** -130]),
    ]).astype(np.float32)
    h = np.resize(vals, (64, 128)).astype(np.float32)
    for fmt, scale in PAIRS:
        st, A, D, _, _, _ = mamba2_from_workload(w, DEV, bd.RSSM_F32, read_copy=False)
        st.ckpt[0, 0].copy_(torch.from_numpy(h))
        err, ws = emu_buffers(st)
        want = rc.emulate_read(h, fmt, scale)
        got = np.zeros_like(want)
        rec = I.mamba2_step_inputs(w, 0, DEV)
        rec["dt"].fill_(1e-30)            # exp(dt A) = 1 and the window term ~ 0
        rec["z"].fill_(30.0)              # silu(30) = 30 (to 1e-12)
        rec["x"].zero_()
        y = st.new_output()
        for col in range(128):
            st.cursors.zero_()
            C = torch.zeros_like(rec["C"])
            C[0, 0, col] = 1.0
            rec["C"] = C
            st.step_emulated(rec, A, D, y, bd.emulation(FMT[fmt], SCALE[scale]), err, ws)
            got[:, col] = y[0, 0].double().cpu().numpy() / 30.0
        np.testing.assert_allclose(got, want, rtol=2e-7, atol=0, err_msg=f"{fmt}-{scale}")


@pytest.mark.parametrize("batch", [257, 513])
def test_error_report_with_a_ragged_last_chunk(batch):
    """The error report's two-stage reduction over one (error, norm) pair per
    block: a launch of 257 blocks leaves a last chunk of one pair (read as
    the pair itself), 513 blocks a last chunk of one pair after two full
    ones. The report equals the oracle's emulation_error summed over every
    sequence whose step does not flush (<= 1e-5 relative)."""
    w = W("emu_ragged", batch, 1, 64, 128, 1, 4, 3, seed=605)
    st, A, D, _, _, _ = mamba2_from_workload(w, DEV, bd.RSSM_F32, read_copy=False)
    err, ws = emu_buffers(st)
    emu = bd.emulation(FMT["e4m3"], SCALE["tile64"])
    y = st.new_output()
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, DEV)
        counts = st.cursors[:, 1].cpu().numpy()
        h0 = st.ckpt.cpu().numpy()
        e_exp = n_exp = 0.0
        for b in range(w.batch):
            if counts[b] + 1 != w.buf_len:  # a flushing step reads the exact checkpoint
                e, n = rc.emulation_error(h0[b], "e4m3", "tile64")
                e_exp, n_exp = e_exp + e, n_exp + n
        st.step_emulated(rec, A, D, y, emu, err, ws)
        e_gpu, n_gpu = err.tolist()
        assert n_gpu == pytest.approx(n_exp, rel=TOL_ERR), t
        assert e_gpu == pytest.approx(e_exp, rel=TOL_ERR, abs=1e-30), t
    assert H.status(st) == 0
