"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (bf16 outputs; fp32 outputs in one case), on EVERY sequence of the
batch: the fp64 oracle's sessions run in one spawned worker per host core
(tests/oracle_workers.py), each over a chunk of sequences, fed the GPU's
records and outputs step by step.

Checked at every step: each output against the oracle's (bf16: the error
beyond half a bf16 ulp <= 2e-3 x output RMS; fp32: <= 1e-4 relative L2), the
cursors of the whole batch bit-exact against the cursor model, and that a
step writes no checkpoint outside a flush (or a verify outside a fold); at
the end, every sequence's checkpoint against the oracle's state at its last
flush or fold (<= 1e-5 relative L2), or bit-identical to its initial value if
it never flushed. Source: "ReplaySSM Caches Inputs Instead of State...",
section "How ReplaySSM works" (outputs match conventional decoding up to
floating-point differences; the checkpoint is written only by a flush).
"""
import numpy as np
import pytest
import torch

import harness as H
import oracle_workers as OW
from oracle import cursors as oc
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.state import gdn_from_workload, kda_from_workload, mamba2_from_workload

pytestmark = pytest.mark.gpu

TOL_Y32, TOL_CKPT, TOL_BF16_EXCESS, TOL_READ_COPY, TOL_READ_F8 = 1e-4, 1e-5, 2e-3, 1e-2, 2.0 ** -4
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def np32(t):
    """A GPU tensor as fp32 numpy (bf16 widens exactly)."""
    return t.detach().float().cpu().numpy()


def sl(c):
    return slice(int(c[0]), int(c[-1]) + 1)


def host(rec):
    return {k: np32(v) for k, v in rec.items()}


def init_fn(h0, pre, starts, counts, L, **params):
    """The worker's initial data for a chunk (numpy views are pickled per chunk)."""
    h0, pre = np32(h0), host(pre)
    starts, counts = starts.cpu().numpy(), counts.cpu().numpy()

    def init_of(c):
        s = sl(c)
        return dict(h0=h0[s], prefill={k: v[s] for k, v in pre.items()}, starts=starts[s], counts=counts[s], L=L,
                    **params)
    return init_of


def check_outputs(rel, excess, finite, kind):
    for t, (r, e, f) in enumerate(zip(rel, excess, finite)):
        if r is None:
            continue
        assert f, (t, "non-finite output")
        if kind == "bf16":
            assert e <= TOL_BF16_EXCESS, (t, e)
        elif kind == "f32":
            assert r <= TOL_Y32, (t, r)
        else:
            assert r <= kind, (t, r)


def check_checkpoints(ck, ckpt, ckpt0, batch):
    assert all(e <= TOL_CKPT for e in ck.values()), max(ck.items(), key=lambda kv: kv[1])
    never = [b for b in range(batch) if b not in ck]
    if never:
        assert torch.equal(ckpt[never], ckpt0[never])
    return len(ck)


def run_mamba2_ar(w, out_dtype, steps, read_copy=None, compare_steps=None, sample=None, emu=None, reports=None):
    """AR decode of workload w on the GPU beside the oracle pool; returns
    (per-step rel-L2, bf16 excess, finite flags, checkpoint errors, state).
    emu: an emulated read precision (rssm_mamba2_step_emulated), whose
    per-step error reports are appended to ``reports``."""
    st, A, D, pre, starts, counts = mamba2_from_workload(w, DEV, out_dtype, False if emu else read_copy)
    if emu is not None:
        err = torch.zeros(2, dtype=torch.float64, device=DEV)
        ws = torch.empty(bd.rssm_mamba2_emulated_workspace_bytes(st.desc), dtype=torch.uint8, device=DEV)
    ckpt0 = st.ckpt.clone()
    seqs = np.arange(w.batch) if sample is None else np.asarray(sample)
    chunks = OW.chunks_of(len(seqs)) if sample is None else [np.array([i]) for i in range(len(seqs))]
    sel = torch.as_tensor(seqs, device=DEV)
    init_of = init_fn(st.ckpt[sel], {k: v[sel] for k, v in pre.items()}, starts[sel], counts[sel], w.buf_len,
                      A=np32(A), D=np32(D))
    pool = OW.OraclePool("mamba2_ar", chunks, init_of)
    try:
        model = [(int(s), int(c), 0, 0) for s, c in zip(starts.cpu(), counts.cpu())]
        y = st.new_output()
        for t in range(steps):
            rec = I.mamba2_step_inputs(w, t, DEV)
            prev = st.ckpt.clone()
            if emu is None:
                st.step(rec, A, D, y)
            else:
                st.step_emulated(rec, A, D, y, emu, err, ws)
                reports.append(err.tolist())
            model_next = [oc.ar_step(c, w.buf_len) for c in model]
            np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array([m[0] for m in model_next]))
            quiet = [b for b, m in enumerate(model_next) if not m[2]]
            assert torch.equal(st.ckpt[quiet], prev[quiet]), t  # non-flush steps write no state
            model = [m[0] for m in model_next]
            rh = host({k: v[sel] for k, v in rec.items()})
            yh = np32(y[sel]) if compare_steps is None or t < compare_steps else None
            pool.step(lambda c: {k: v[sl(c)] for k, v in rh.items()}, None,
                      None if yh is None else (lambda c: yh[sl(c)]))
        ck = np32(st.ckpt[sel])
        rel, excess, finite, cke = pool.finish(lambda c: ck[sl(c)])
    finally:
        pool.close()
    assert H.status(st) == 0
    return rel, excess, finite, {int(seqs[i]): e for i, e in cke.items()}, st, ckpt0


def test_mamba2_serving_full_size():
    """Batch 256, 128 heads, 64x128 state, 8 groups, L=16, staggered windows,
    256 steps, bf16 outputs: all 256 sequences at every step."""
    w = I.WORKLOADS["mamba2_serving"]
    rel, excess, finite, ck, st, ckpt0 = run_mamba2_ar(w, bd.RSSM_BF16, w.steps)
    check_outputs(rel, excess, finite, "bf16")
    assert check_checkpoints(ck, st.ckpt, ckpt0, w.batch) == w.batch   # every sequence flushed


def test_mamba2_serving_fp32_outputs():
    """The same layer with fp32 outputs, 256 steps, all sequences, 1e-4 rel-L2."""
    w = I.WORKLOADS["mamba2_serving"]
    rel, excess, finite, ck, st, ckpt0 = run_mamba2_ar(w, bd.RSSM_F32, w.steps)
    check_outputs(rel, excess, finite, "f32")
    assert check_checkpoints(ck, st.ckpt, ckpt0, w.batch) == w.batch


def run_spec(kind, w, st, verify, rec_fn, steps, init_of, ckpt_of, state_tensor, out):
    """Speculative decode on the GPU beside the oracle pool (every sequence)."""
    ckpt0 = state_tensor.clone()
    pool = OW.OraclePool(kind, OW.chunks_of(w.batch), init_of)
    try:
        model = [tuple(int(v) for v in c) for c in st.cursors.cpu()]
        folds = 0
        for t in range(steps):
            rec = rec_fn(w, t, DEV)
            kept = I.accepted_kept(w, t, DEV)
            prev = state_tensor.clone()
            verify(rec, out)
            mv = [oc.verify(c, w.n_new, w.buf_len) for c in model]
            np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array([m[0] for m in mv]))
            quiet = [b for b, m in enumerate(mv) if not m[2]]
            assert torch.equal(state_tensor[quiet], prev[quiet]), t  # only a folding verify writes the checkpoint
            folds += len(mv) - len(quiet)
            st.commit(kept)
            kl = kept.cpu().tolist()
            model = [oc.commit(m[0], k, w.buf_len)[0] for m, k in zip(mv, kl)]
            np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array(model))
            rh, kh, oh = host(rec), kept.cpu().numpy(), np32(out)
            pool.step(lambda c: {k: v[sl(c)] for k, v in rh.items()}, lambda c: kh[sl(c)], lambda c: oh[sl(c)])
        rel, excess, finite, ck = pool.finish(ckpt_of)
    finally:
        pool.close()
    assert folds > 0
    assert H.status(st) == 0
    return rel, excess, finite, ck, ckpt0


SPEC_VERIFIES = 48  # six window cycles of 8 verifies (K = 4, L = 16), every sequence checked


def test_mamba2_spec_full_size():
    """Batch 512, K = 4 records per verify, accepted ~U{0..3}, flush on
    overflow; 48 verifies, all 512 sequences."""
    w = I.WORKLOADS["mamba2_spec"]
    st, A, D, pre, starts, counts = mamba2_from_workload(w, DEV, bd.RSSM_BF16)
    init_of = init_fn(st.ckpt, pre, starts, counts, w.buf_len, A=np32(A), D=np32(D))
    y = st.new_output(w.n_new)
    final = {}

    def ckpt_of(c):
        if "ck" not in final:
            final["ck"] = np32(st.ckpt)
        return final["ck"][sl(c)]

    rel, excess, finite, ck, ckpt0 = run_spec("mamba2_spec", w, st, lambda r, o: st.verify(r, A, D, o),
                                             I.mamba2_verify_inputs, SPEC_VERIFIES, init_of, ckpt_of, st.ckpt, y)
    check_outputs(rel, excess, finite, "bf16")
    assert check_checkpoints(ck, st.ckpt, ckpt0, w.batch) > w.batch // 2


def run_delta_ar(kind, w, setup, rec_fn):
    st, pre, starts, counts = setup(w, DEV, bd.RSSM_BF16)
    S0 = st.S.clone()
    init_of = init_fn(st.S, pre, starts, counts, w.buf_len)
    pool = OW.OraclePool(kind, OW.chunks_of(w.batch), init_of)
    try:
        model = [(int(s), int(c), 0, 0) for s, c in zip(starts.cpu(), counts.cpu())]
        o = st.new_output()
        for t in range(w.steps):
            rec = rec_fn(w, t, DEV)
            prev = st.S.clone()
            st.step(rec, o)
            mn = [oc.ar_step(c, w.buf_len) for c in model]
            np.testing.assert_array_equal(st.cursors.cpu().numpy(), np.array([m[0] for m in mn]))
            quiet = [b for b, m in enumerate(mn) if not m[2]]
            assert torch.equal(st.S[quiet], prev[quiet]), t
            model = [m[0] for m in mn]
            rh, oh = host(rec), np32(o)
            pool.step(lambda c: {k: v[sl(c)] for k, v in rh.items()}, None, lambda c: oh[sl(c)])
        sh = np32(st.S)
        rel, excess, finite, ck = pool.finish(lambda c: sh[sl(c)])
    finally:
        pool.close()
    assert H.status(st) == 0
    check_outputs(rel, excess, finite, "bf16")
    assert check_checkpoints(ck, st.S, S0, w.batch) == w.batch


def test_gdn_serving_full_size():
    """Batch 256, 32 heads, 128x128 state, L=16, staggered windows, 256 steps, all sequences."""
    run_delta_ar("gdn_ar", I.WORKLOADS["gdn_serving"], gdn_from_workload, I.gdn_step_inputs)


def test_kda_serving_full_size():
    """Kimi Delta Attention at the bench's size: batch 256, 32 heads, 128x128
    state, L=16, staggered windows, 256 steps, all sequences."""
    run_delta_ar("kda_ar", I.WORKLOADS["kda_serving"], kda_from_workload, I.kda_step_inputs)


@pytest.mark.parametrize("name", ["gdn_spec", "kda_spec"])
def test_delta_spec_full_size(name):
    """Gated DeltaNet (and KDA) speculative decode: batch 512, 32 heads,
    128x128 state, K = 4 records per verify, accepted ~U{0..3}, fold on
    overflow; 48 verifies, all 512 sequences."""
    w = I.WORKLOADS[name]
    setup, rec_fn = ((gdn_from_workload, I.gdn_verify_inputs) if name == "gdn_spec"
                     else (kda_from_workload, I.kda_verify_inputs))
    st, pre, starts, counts = setup(w, DEV, bd.RSSM_BF16)
    init_of = init_fn(st.S, pre, starts, counts, w.buf_len)
    o = st.new_verify_output(w.n_new)
    final = {}

    def ckpt_of(c):
        if "ck" not in final:
            final["ck"] = np32(st.S)
        return final["ck"][sl(c)]

    kind = "gdn_spec" if name == "gdn_spec" else "kda_spec"
    rel, excess, finite, ck, S0 = run_spec(kind, w, st, st.verify, rec_fn, SPEC_VERIFIES, init_of, ckpt_of, st.S, o)
    check_outputs(rel, excess, finite, "bf16")
    assert check_checkpoints(ck, st.S, S0, w.batch) > w.batch // 2


def spread(counts, n):
    """n sequence indices spanning the range of initial window counts."""
    order = np.argsort(counts.cpu().numpy(), kind="stable")
    idx = np.linspace(0, len(order) - 1, n).round().astype(int)
    return sorted(set(int(order[i]) for i in idx))


@pytest.mark.parametrize("name", ["mamba2_bf16_read", "mamba2_f16_read", "mamba2_f8_read"])
def test_read_copy_all_sequences(name):
    """fp32 recurrence checkpoint + bf16 / fp16 / fp8 read copy, all 256
    sequences over four window cycles (64 steps): outputs within 1e-2
    relative L2 (2^-4, the e4m3 half-ulp, for fp8), checkpoints at 1e-5, and
    the read copy of every sequence equal, bit for bit, to the oracle's
    rounding of its fp32 checkpoint."""
    w = I.WORKLOADS[name]
    rel, excess, finite, ck, st, ckpt0 = run_mamba2_ar(w, bd.RSSM_F32, 64)
    check_outputs(rel, excess, finite, TOL_READ_F8 if w.read_copy == "f8" else TOL_READ_COPY)
    assert check_checkpoints(ck, st.ckpt, ckpt0, w.batch) == w.batch
    for b in range(0, w.batch, 8):
        H.assert_read_copy(st, b)


@pytest.mark.parametrize("name", ["mamba2_bf16_read", "mamba2_f16_read", "mamba2_f8_read"])
def test_read_copy_4096_steps(name):
    """The same layer over 4096 steps, on 16 sequences spanning the initial
    window counts (one oracle worker each): the output error stays within the
    bound and does not grow (rounding of the read copy never enters the
    recurrence)."""
    w = I.WORKLOADS[name]
    sample = spread(I.initial_cursors(w, DEV)[1], 16)
    rel, excess, finite, ck, st, ckpt0 = run_mamba2_ar(w, bd.RSSM_F32, w.steps, sample=sample)
    trace = np.array(rel)
    assert all(finite)
    assert trace.max() <= (TOL_READ_F8 if w.read_copy == "f8" else TOL_READ_COPY)
    assert trace[-512:].max() <= 1.25 * trace[:512].max()
    slope = np.polyfit(np.arange(len(trace)), trace, 1)[0]
    assert slope < 1e-7, slope
    assert all(e <= TOL_CKPT for e in ck.values())


@pytest.mark.parametrize("fmt", ["e4m3", "int8"])
def test_emulated_read_4096_steps(fmt):
    """The serving layer with an emulated read precision (one scale per 64-row
    tile: e4m3, or int8), 4096 steps, 16 sequences spanning the initial window
    counts: the output error against the fp64 conventional decode stays within
    the read's own bound (e4m3: 2^-4; int8: 2^-6, half an int8 step of a tile
    whose largest element is about 4 of its RMS) and does not grow, and the
    error each call reports stays at a constant level."""
    w = I.WORKLOADS["mamba2_serving"]
    w = type(w)(**{**w.__dict__, "name": "mamba2_emu", "steps": 4096})
    emu = bd.emulation(bd.RSSM_EMU_E4M3 if fmt == "e4m3" else bd.RSSM_EMU_INT8, bd.RSSM_EMU_SCALE_TILE64)
    sample = spread(I.initial_cursors(w, DEV)[1], 16)
    reports = []
    rel, excess, finite, ck, st, ckpt0 = run_mamba2_ar(w, bd.RSSM_F32, w.steps, sample=sample, emu=emu,
                                                      reports=reports)
    trace = np.array(rel)
    assert all(finite)
    assert trace.max() <= (2.0 ** -4 if fmt == "e4m3" else 2.0 ** -6), trace.max()
    assert trace[-512:].max() <= 1.25 * trace[:512].max()
    assert np.polyfit(np.arange(len(trace)), trace, 1)[0] < 1e-7
    assert all(e <= TOL_CKPT for e in ck.values())
    q = np.sqrt([e / n for e, n in reports])     # relative L2 error of each call's emulated read
    assert q[-512:].max() <= 1.25 * q[:512].max() and q.min() > 0
