"""The serving boundary against the oracle: decode calls made through a state
slot table (a permuted batch with padding rows) and calls replayed from a
CUDA graph, compared with the fp64 oracle's decode sessions of the same
sequences -- outputs, the checkpoint of every sequence that flushed or folded
(and its read copy, bit for bit), and the cursors (bit-exact).

Source: "ReplaySSM" (the paper's code repository), the paragraph on the vLLM
integration (metadata and dispatch around the kernels); a slot call computes
the same quantities as any other call ("ReplaySSM Caches Inputs Instead of
State...", section "How ReplaySSM works": outputs match conventional decoding
up to floating-point differences).
"""
import numpy as np
import pytest
import torch

import harness as H
from oracle import sessions
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import GDNWorkload as GW
from recurrent_state_decode_gb300.inputs import KDAWorkload as KW
from recurrent_state_decode_gb300.inputs import Mamba2Workload as W
from recurrent_state_decode_gb300.state import (GDNState, KDAState, Mamba2State, gdn_from_workload,
                                                kda_from_workload, mamba2_from_workload)

pytestmark = pytest.mark.gpu

TOL_Y32, TOL_CKPT, TOL_BF16_EXCESS, TOL_READ_COPY, TOL_READ_F8 = 1e-4, 1e-5, 2e-3, 1e-2, 2.0 ** -4

PERM = [5, 0, 3]      # state slot of sequence b
ROWS = 5              # batch rows of a slot call
ROW_OF = [2, 4, 1]    # batch row of sequence b
PAD = [0, 3]          # padding rows
N_SLOTS = 7           # state rows; 1, 2, 4, 6 are named by no row
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def slot_table():
    t = torch.full((ROWS,), -1, dtype=torch.int32, device=DEV)
    t[ROW_OF] = torch.tensor(PERM, dtype=torch.int32, device=DEV)
    return t


def rows_of(rec):
    """The slot call's records: sequence b at row ROW_OF[b]; padding rows hold
    sequence 0's values (never read)."""
    out = {}
    for k, v in rec.items():
        r = v[[0] * ROWS].clone()
        r[ROW_OF] = v
        out[k] = r
    return out


def kept_rows(kept):
    k = torch.full((ROWS,), 999, dtype=torch.int32, device=DEV)  # padding rows: a kept no commit may apply
    k[ROW_OF] = kept
    return k


def place(plain, slotted, fields):
    """Copy the plain session's state rows into slots PERM of a state whose
    other rows hold random values; returns the untouched rows' snapshot."""
    g = torch.Generator(device=DEV).manual_seed(17)
    for f in fields:
        t = getattr(slotted, f)
        if t.dtype in (torch.int32, torch.uint8):
            t.copy_(torch.randint(0, 100, t.shape, generator=g, device=DEV, dtype=torch.int32).to(t.dtype))
        else:
            t.copy_(torch.randn(t.shape, generator=g, device=DEV).to(t.dtype))
        t[PERM] = getattr(plain, f)
    unused = [s for s in range(N_SLOTS) if s not in PERM]
    return unused, {f: getattr(slotted, f)[unused].clone() for f in fields}


def check_untouched(st, unused, snap):
    for f, v in snap.items():
        assert torch.equal(getattr(st, f)[unused], v), f + ": a state row no batch row names"


def check_out(y, ref, kind):
    yg = H.F64(y)
    if kind == "f32":
        assert H.rel_l2(yg, ref) <= TOL_Y32
    elif kind == "bf16":
        assert H.bf16_excess(yg, ref) <= TOL_BF16_EXCESS
    else:
        assert H.rel_l2(yg, ref) <= (TOL_READ_F8 if kind == "f8" else TOL_READ_COPY)


M2_FIELDS = ("ckpt", "rx", "rz", "rB", "rC", "rdt", "cursors")


def m2_slotted(w, read_copy, out_dtype):
    sa, A, D, pre, starts, counts = mamba2_from_workload(w, DEV, out_dtype, read_copy)
    ss = Mamba2State(N_SLOTS, w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len, DEV, read_copy=read_copy,
                     out_dtype=out_dtype)
    fields = M2_FIELDS + ((("read_q", "read_scale") if read_copy == "f8" else ("ckpt_read",)) if read_copy else ())
    unused, snap = place(sa, ss, fields)
    return sa, ss, A, D, pre, starts, counts, unused, snap


def out_kind(out_dtype, read_copy):
    if read_copy:
        return "f8" if read_copy == "f8" else "rc"
    return "bf16" if out_dtype == bd.RSSM_BF16 else "f32"


@pytest.mark.parametrize("read_copy,out_dtype", [(False, bd.RSSM_F32), (False, bd.RSSM_BF16), (True, bd.RSSM_F32),
                                                 ("f16", bd.RSSM_F32), ("f8", bd.RSSM_F32)],
                         ids=["f32", "bf16out", "bf16read", "f16read", "f8read"])
def test_mamba2_step_with_slots_against_the_oracle(read_copy, out_dtype):
    # 8 heads in 2 groups (4 heads share a ring group row), L = 8, 20 steps:
    # every sequence flushes at least twice, from staggered windows
    w = W("so_m2", 3, 8, 64, 128, 2, 8, 20, seed=501)
    sa, ss, A, D, pre, starts, counts, unused, snap = m2_slotted(w, read_copy, out_dtype)
    feed = H.Feed()
    sess = sessions.mamba2_ar_session(H.F64(sa.ckpt), H.sub(pre, slice(None)), starts.cpu().numpy(),
                                      counts.cpu().numpy(), feed, H.F64(A), H.F64(D), w.buf_len)
    del sa
    slots = slot_table()
    kind = out_kind(out_dtype, read_copy)
    flushes = 0
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, DEV)
        feed.rec = H.sub(rec, slice(None))
        y = torch.full((ROWS, w.nheads, w.headdim), float("nan"), device=DEV).to(ss.y_dtype)
        ss.step(rows_of(rec), A, D, y, slots=slots)
        exp = next(sess)
        check_out(y[ROW_OF], exp["y"], kind)
        assert torch.isnan(y[PAD]).all(), t
        np.testing.assert_array_equal(ss.cursors[PERM].cpu().numpy(), exp["cursors"])
        for b in np.nonzero(exp["flushed"])[0]:
            flushes += 1
            assert H.rel_l2(H.F64(ss.ckpt[PERM[b]]), exp["state"][b]) <= TOL_CKPT, (t, b)
            if read_copy:
                H.assert_read_copy(ss, PERM[b])
    assert flushes >= 2 * w.batch
    check_untouched(ss, unused, snap)
    assert H.status(ss) == 0


@pytest.mark.parametrize("read_copy", [False, "f8"], ids=["f32", "f8read"])
def test_mamba2_verify_commit_with_slots_against_the_oracle(read_copy):
    w = W("so_m2_spec", 3, 8, 64, 128, 2, 8, 12, seed=502, drafts=3)
    sa, ss, A, D, pre, starts, counts, unused, snap = m2_slotted(w, read_copy, bd.RSSM_F32)
    fv, fk = H.Feed(), H.Feed()
    sess = sessions.mamba2_spec_session(H.F64(sa.ckpt), H.sub(pre, slice(None)), starts.cpu().numpy(),
                                        counts.cpu().numpy(), fv, fk, H.F64(A), H.F64(D), w.buf_len)
    del sa
    slots = slot_table()
    kind = out_kind(bd.RSSM_F32, read_copy)
    folds = 0
    for t in range(w.steps):
        rec = I.mamba2_verify_inputs(w, t, DEV)
        kept = I.accepted_kept(w, t, DEV)
        fv.rec, fk.rec = H.sub(rec, slice(None)), kept.cpu().numpy()
        y = torch.full((ROWS, w.n_new, w.nheads, w.headdim), float("nan"), device=DEV)
        ss.verify(rows_of(rec), A, D, y, slots=slots)
        cv = ss.cursors[PERM].cpu().numpy()
        ss.commit(kept_rows(kept), slots=slots)
        exp = next(sess)
        check_out(y[ROW_OF], exp["y"], kind)
        assert torch.isnan(y[PAD]).all(), t
        np.testing.assert_array_equal(cv, exp["cursors_verify"])
        np.testing.assert_array_equal(ss.cursors[PERM].cpu().numpy(), exp["cursors_commit"])
        for b in np.nonzero(exp["folded"])[0]:
            folds += 1
            assert H.rel_l2(H.F64(ss.ckpt[PERM[b]]), exp["committed_state"][b]) <= TOL_CKPT, (t, b)
            if read_copy:
                H.assert_read_copy(ss, PERM[b])
    assert folds > 0
    check_untouched(ss, unused, snap)
    assert H.status(ss) == 0


GDN_FIELDS = ("S", "rq", "rk", "rv", "rg", "rbeta", "re", "cursors")


@pytest.mark.parametrize("kda", [False, True], ids=["gdn", "kda"])
def test_delta_step_with_slots_against_the_oracle(kda):
    if kda:
        w = KW("so_kda", 3, 2, 128, 128, 8, 20, seed=503)
        sa, pre, starts, counts = kda_from_workload(w, DEV)
        ss = KDAState(N_SLOTS, w.nheads, w.dk, w.dv, w.buf_len, DEV)
        session, step_inputs = sessions.kda_ar_session, I.kda_step_inputs
    else:
        w = GW("so_gdn", 3, 2, 128, 128, 8, 20, seed=504)
        sa, pre, starts, counts = gdn_from_workload(w, DEV)
        ss = GDNState(N_SLOTS, w.nheads, w.dk, w.dv, w.buf_len, DEV)
        session, step_inputs = sessions.gdn_ar_session, I.gdn_step_inputs
    unused, snap = place(sa, ss, GDN_FIELDS)
    feed = H.Feed()
    sess = session(H.F64(sa.S), H.sub(pre, slice(None)), starts.cpu().numpy(), counts.cpu().numpy(), feed,
                   w.buf_len)
    del sa
    slots = slot_table()
    flushes = 0
    for t in range(w.steps):
        rec = step_inputs(w, t, DEV)
        feed.rec = H.sub(rec, slice(None))
        o = torch.full((ROWS, w.nheads, w.dv), float("nan"), device=DEV)
        ss.step(rows_of(rec), o, slots=slots)
        exp = next(sess)
        check_out(o[ROW_OF], exp["o"], "f32")
        assert torch.isnan(o[PAD]).all(), t
        np.testing.assert_array_equal(ss.cursors[PERM].cpu().numpy(), exp["cursors"])
        for b in np.nonzero(exp["flushed"])[0]:
            flushes += 1
            assert H.rel_l2(H.F64(ss.S[PERM[b]]), exp["state"][b]) <= TOL_CKPT, (t, b)
    assert flushes >= 2 * w.batch
    check_untouched(ss, unused, snap)
    assert H.status(ss) == 0


@pytest.mark.parametrize("kda", [False, True], ids=["gdn", "kda"])
def test_delta_verify_commit_with_slots_against_the_oracle(kda):
    if kda:
        w = KW("so_kda_spec", 3, 2, 128, 128, 8, 12, seed=506, drafts=3)
        sa, pre, starts, counts = kda_from_workload(w, DEV)
        ss = KDAState(N_SLOTS, w.nheads, w.dk, w.dv, w.buf_len, DEV)
        session, verify_inputs = sessions.kda_spec_session, I.kda_verify_inputs
    else:
        w = GW("so_gdn_spec", 3, 2, 128, 128, 8, 12, seed=505, drafts=3)
        sa, pre, starts, counts = gdn_from_workload(w, DEV)
        ss = GDNState(N_SLOTS, w.nheads, w.dk, w.dv, w.buf_len, DEV)
        session, verify_inputs = sessions.gdn_spec_session, I.gdn_verify_inputs
    unused, snap = place(sa, ss, GDN_FIELDS)
    fv, fk = H.Feed(), H.Feed()
    sess = session(H.F64(sa.S), H.sub(pre, slice(None)), starts.cpu().numpy(), counts.cpu().numpy(), fv, fk,
                   w.buf_len)
    del sa
    slots = slot_table()
    folds = 0
    for t in range(w.steps):
        rec = verify_inputs(w, t, DEV)
        kept = I.accepted_kept(w, t, DEV)
        fv.rec, fk.rec = H.sub(rec, slice(None)), kept.cpu().numpy()
        o = torch.full((ROWS, w.n_new, w.nheads, w.dv), float("nan"), device=DEV)
        ss.verify(rows_of(rec), o, slots=slots)
        cv = ss.cursors[PERM].cpu().numpy()
        ss.commit(kept_rows(kept), slots=slots)
        exp = next(sess)
        check_out(o[ROW_OF], exp["o"], "f32")
        assert torch.isnan(o[PAD]).all(), t
        np.testing.assert_array_equal(cv, exp["cursors_verify"])
        np.testing.assert_array_equal(ss.cursors[PERM].cpu().numpy(), exp["cursors_commit"])
        for b in np.nonzero(exp["folded"])[0]:
            folds += 1
            assert H.rel_l2(H.F64(ss.S[PERM[b]]), exp["committed_state"][b]) <= TOL_CKPT, (t, b)
    assert folds > 0
    check_untouched(ss, unused, snap)
    assert H.status(ss) == 0


def _graph(fn):
    """Capture fn() into a CUDA graph on a side stream (nothing runs) and return it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


def test_graph_replay_with_slots_against_the_oracle():
    """Twelve Mamba-2 slot steps captured once with an all-padding slot table,
    the real table written afterwards, one replay: every step's outputs, the
    flushed checkpoints and the cursors against the oracle's session."""
    w = W("so_graph", 3, 8, 64, 128, 2, 8, 12, seed=506)
    sa, ss, A, D, pre, starts, counts, unused, snap = m2_slotted(w, False, bd.RSSM_F32)
    h0 = H.F64(sa.ckpt)
    del sa
    recs = [rows_of(I.mamba2_step_inputs(w, t, DEV)) for t in range(w.steps)]
    ys = [torch.full((ROWS, w.nheads, w.headdim), float("nan"), device=DEV) for _ in range(w.steps)]
    slots = torch.full((ROWS,), -1, dtype=torch.int32, device=DEV)

    def steps():
        for t in range(w.steps):
            ss.step(recs[t], A, D, ys[t], slots=slots)

    g = _graph(steps)
    slots.copy_(slot_table())
    g.replay()
    torch.cuda.synchronize()
    sess = sessions.mamba2_ar_session(h0, H.sub(pre, slice(None)), starts.cpu().numpy(), counts.cpu().numpy(),
                                      ({k: H.F64(v[ROW_OF]) for k, v in r.items()} for r in recs),
                                      H.F64(A), H.F64(D), w.buf_len)
    last_state = {}
    for t in range(w.steps):
        exp = next(sess)
        check_out(ys[t][ROW_OF], exp["y"], "f32")
        assert torch.isnan(ys[t][PAD]).all(), t
        for b in np.nonzero(exp["flushed"])[0]:
            last_state[b] = exp["state"][b]
    np.testing.assert_array_equal(ss.cursors[PERM].cpu().numpy(), exp["cursors"])
    assert last_state, "some sequence flushed"
    for b, s in last_state.items():  # the checkpoint holds the state at its latest flush
        assert H.rel_l2(H.F64(ss.ckpt[PERM[b]]), s) <= TOL_CKPT, b
    check_untouched(ss, unused, snap)
    assert H.status(ss) == 0


def test_graph_replay_gdn_verify_against_the_oracle():
    """Gated DeltaNet verify + commit steps captured in one graph (no slots),
    replayed once, against the oracle's speculative session."""
    w = GW("so_graph_gdn", 3, 2, 128, 128, 8, 8, seed=507, drafts=3)
    st, pre, starts, counts = gdn_from_workload(w, DEV)
    S0 = H.F64(st.S)
    recs = [I.gdn_verify_inputs(w, t, DEV) for t in range(w.steps)]
    kepts = [I.accepted_kept(w, t, DEV) for t in range(w.steps)]
    outs = [st.new_verify_output(w.n_new) for _ in range(w.steps)]

    def steps():
        for t in range(w.steps):
            st.verify(recs[t], outs[t])
            st.commit(kepts[t])

    g = _graph(steps)
    g.replay()
    torch.cuda.synchronize()
    sess = sessions.gdn_spec_session(S0, H.sub(pre, slice(None)), starts.cpu().numpy(), counts.cpu().numpy(),
                                     (H.sub(r, slice(None)) for r in recs), (k.cpu().numpy() for k in kepts),
                                     w.buf_len)
    for t in range(w.steps):
        exp = next(sess)
        check_out(outs[t], exp["o"], "f32")
    np.testing.assert_array_equal(st.cursors.cpu().numpy(), exp["cursors_commit"])
    assert H.status(st) == 0
