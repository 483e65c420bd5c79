"""State slots: decode calls whose batch rows use state rows named by a slot
table, with padding rows (slot -1) skipped.

A slot call runs the same kernels on the same values as a call without slots,
so it must reproduce one bit for bit: every sequence's outputs, checkpoint,
read copy, ring and cursor; padding rows leave their outputs unwritten; state
rows that no batch row names are left untouched; a slot outside the state
arrays is reported (RSSM_DEV_BAD_SLOT) and its row skipped while the other
rows still run.
"""
import pytest
import torch

import harness as H
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import GDNWorkload as GW
from recurrent_state_decode_gb300.inputs import Mamba2Workload as W
from recurrent_state_decode_gb300.state import GDNState, Mamba2State

pytestmark = pytest.mark.gpu

PERM = [5, 0, 3]                 # state slot of sequence b
ROWS = 5                         # batch rows of a slot call
ROW_OF = [2, 4, 1]               # batch row of sequence b
PAD = [0, 3]                     # padding rows
N_SLOTS = 7                      # state rows; slots 1, 2, 4, 6 are named by no row


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def _slot_table(dev, bad=None):
    t = torch.full((ROWS,), -1, dtype=torch.int32, device=dev)
    for b, r in enumerate(ROW_OF):
        t[r] = PERM[b]
    if bad is not None:  # (row, slot): a padding row naming a slot outside the state arrays
        t[bad[0]] = bad[1]
    return t


def _rows(rec, fill=None):
    """Records of the slot call: sequence b's at row ROW_OF[b]; padding rows hold
    sequence 0's values (never read)."""
    out = {}
    for k, v in rec.items():
        r = v[[0] * ROWS].clone() if fill is None else torch.full((ROWS,) + tuple(v.shape[1:]), fill,
                                                                  dtype=v.dtype, device=v.device)
        r[ROW_OF] = v
        out[k] = r
    return out


def _m2_fields(st):
    f = {"ckpt": st.ckpt, "rx": st.rx, "rz": st.rz, "rB": st.rB, "rC": st.rC, "rdt": st.rdt,
         "cursors": st.cursors}
    if st.ckpt_read is not None:
        if hasattr(st, "read_q"):
            f["read_q"], f["read_scale"] = st.read_q, st.read_scale
        else:
            f["ckpt_read"] = st.ckpt_read
    return f


def _gdn_fields(st):
    return {"S": st.S, "rq": st.rq, "rk": st.rk, "rv": st.rv, "rg": st.rg, "rbeta": st.rbeta, "re": st.re,
            "cursors": st.cursors}


def _fill_random(fields, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    for name, t in fields.items():
        if t.dtype in (torch.int32, torch.uint8):
            t.copy_(torch.randint(0, 100, t.shape, generator=g, device=t.device, dtype=torch.int32).to(t.dtype))
        else:
            t.copy_(torch.randn(t.shape, generator=g, device=t.device).to(t.dtype))


def _place(slot_fields, ref_fields):
    for name, t in slot_fields.items():
        t[PERM] = ref_fields[name]
    unused = [s for s in range(N_SLOTS) if s not in PERM]
    return unused, {name: t[unused].clone() for name, t in slot_fields.items()}


def _check_state(slot_fields, ref_fields, unused, snapshot):
    for name, t in slot_fields.items():
        assert torch.equal(t[PERM], ref_fields[name]), name
        assert torch.equal(t[unused], snapshot[name]), name + " (a state row no batch row names)"


def _m2_pair(w, read_copy, out_dtype=bd.RSSM_F32):
    dev = "cuda"
    sa, A, D, _, _, _ = H.mamba2_setup(w, dev, out_dtype=out_dtype, read_copy=read_copy)
    ss = Mamba2State(N_SLOTS, w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len, dev, read_copy=read_copy,
                     out_dtype=out_dtype)
    _fill_random(_m2_fields(ss), 7)
    unused, snap = _place(_m2_fields(ss), _m2_fields(sa))
    return sa, ss, A, D, unused, snap


@pytest.mark.parametrize("read_copy", [False, True, "f16", "f8"], ids=["f32", "bf16", "f16", "f8"])
def test_mamba2_step_with_slots_matches_the_plain_call(read_copy):
    # L = 8 and 12 steps: flushes on the way, from every starting count of the prefilled windows
    w = W("slots_m2", 3, 4, 64, 128, 2, 8, 12, seed=301)
    sa, ss, A, D, unused, snap = _m2_pair(w, read_copy)
    slots = _slot_table("cuda")
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, "cuda")
        ya = sa.new_output()
        sa.step(rec, A, D, ya)
        ys = torch.full((ROWS, w.nheads, w.headdim), float("nan"), device="cuda")
        ss.step(_rows(rec), A, D, ys, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(ys[ROW_OF], ya), t
        assert torch.isnan(ys[PAD]).all(), t
    _check_state(_m2_fields(ss), _m2_fields(sa), unused, snap)
    assert H.status(sa) == 0 and H.status(ss) == 0


def test_mamba2_step_with_slots_bf16_output_and_group_sharing():
    # 8 heads over 2 groups (4 heads share a group row of the ring), bf16 y
    w = W("slots_m2_g", 3, 8, 128, 128, 2, 5, 7, seed=302)
    sa, ss, A, D, unused, snap = _m2_pair(w, False, bd.RSSM_BF16)
    slots = _slot_table("cuda")
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, "cuda")
        ya = sa.new_output()
        sa.step(rec, A, D, ya)
        ys = ss.new_output(rows=ROWS).fill_(7.0)
        ss.step(_rows(rec), A, D, ys, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(ys[ROW_OF], ya), t
        assert (ys[PAD] == 7.0).all(), t
    _check_state(_m2_fields(ss), _m2_fields(sa), unused, snap)


@pytest.mark.parametrize("read_copy", [False, "f8"], ids=["f32", "f8"])
def test_mamba2_verify_commit_with_slots_matches_the_plain_calls(read_copy):
    w = W("slots_m2_spec", 3, 4, 64, 128, 2, 8, 6, seed=303, drafts=3)
    sa, ss, A, D, unused, snap = _m2_pair(w, read_copy)
    slots = _slot_table("cuda")
    for t in range(w.steps):
        rec = I.mamba2_verify_inputs(w, t, "cuda")
        kept = I.accepted_kept(w, t, "cuda")
        ya = sa.new_output(w.n_new)
        sa.verify(rec, A, D, ya)
        sa.commit(kept)
        ys = torch.full((ROWS, w.n_new, w.nheads, w.headdim), float("nan"), device="cuda")
        ss.verify(_rows(rec), A, D, ys, slots=slots)
        kept_rows = torch.full((ROWS,), 999, dtype=torch.int32, device="cuda")  # padding: would be a bad kept
        kept_rows[ROW_OF] = kept
        ss.commit(kept_rows, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(ys[ROW_OF], ya), t
        assert torch.isnan(ys[PAD]).all(), t
    _check_state(_m2_fields(ss), _m2_fields(sa), unused, snap)
    assert H.status(sa) == 0 and H.status(ss) == 0


def test_mamba2_bad_slot_is_reported_and_skipped():
    w = W("slots_m2_bad", 3, 4, 64, 128, 2, 8, 3, seed=304)
    sa, ss, A, D, unused, snap = _m2_pair(w, False)
    slots = _slot_table("cuda", bad=(0, N_SLOTS))  # padding row 0 names slot 7 of 7
    for t in range(w.steps):
        rec = I.mamba2_step_inputs(w, t, "cuda")
        ya = sa.new_output()
        sa.step(rec, A, D, ya)
        ys = torch.full((ROWS, w.nheads, w.headdim), float("nan"), device="cuda")
        ss.step(_rows(rec), A, D, ys, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(ys[ROW_OF], ya), t
        assert torch.isnan(ys[PAD]).all(), t
    assert H.status(ss) == bd.RSSM_DEV_BAD_SLOT
    _check_state(_m2_fields(ss), _m2_fields(sa), unused, snap)
    # the commit reports a bad slot the same way
    ss.status.zero_()
    kept = torch.zeros(ROWS, dtype=torch.int32, device="cuda")
    ss.commit(kept, slots=_slot_table("cuda", bad=(3, -2)))
    torch.cuda.synchronize()
    assert H.status(ss) == bd.RSSM_DEV_BAD_SLOT


def _gdn_pair(w):
    dev = "cuda"
    sa, _, _, _ = H.gdn_setup(w, dev)
    ss = GDNState(N_SLOTS, w.nheads, w.dk, w.dv, w.buf_len, dev)
    _fill_random(_gdn_fields(ss), 8)
    unused, snap = _place(_gdn_fields(ss), _gdn_fields(sa))
    return sa, ss, unused, snap


def test_gdn_step_with_slots_matches_the_plain_call():
    w = GW("slots_gdn", 3, 2, 128, 128, 8, 12, seed=305)
    sa, ss, unused, snap = _gdn_pair(w)
    slots = _slot_table("cuda")
    for t in range(w.steps):
        rec = I.gdn_step_inputs(w, t, "cuda")
        oa = sa.new_output()
        sa.step(rec, oa)
        os_ = torch.full((ROWS, w.nheads, w.dv), float("nan"), device="cuda")
        ss.step(_rows(rec), os_, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(os_[ROW_OF], oa), t
        assert torch.isnan(os_[PAD]).all(), t
    _check_state(_gdn_fields(ss), _gdn_fields(sa), unused, snap)
    assert H.status(sa) == 0 and H.status(ss) == 0


def test_gdn_verify_commit_with_slots_matches_the_plain_calls():
    w = GW("slots_gdn_spec", 3, 2, 128, 128, 8, 6, seed=306, drafts=3)
    sa, ss, unused, snap = _gdn_pair(w)
    slots = _slot_table("cuda")
    for t in range(w.steps):
        rec = I.gdn_verify_inputs(w, t, "cuda")
        kept = I.accepted_kept(w, t, "cuda")
        oa = sa.new_verify_output(w.n_new)
        sa.verify(rec, oa)
        sa.commit(kept)
        os_ = torch.full((ROWS, w.n_new, w.nheads, w.dv), float("nan"), device="cuda")
        ss.verify(_rows(rec), os_, slots=slots)
        kept_rows = torch.full((ROWS,), 999, dtype=torch.int32, device="cuda")
        kept_rows[ROW_OF] = kept
        ss.commit(kept_rows, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(os_[ROW_OF], oa), t
        assert torch.isnan(os_[PAD]).all(), t
    _check_state(_gdn_fields(ss), _gdn_fields(sa), unused, snap)
    assert H.status(sa) == 0 and H.status(ss) == 0


def test_gdn_bad_slot_is_reported_and_skipped():
    w = GW("slots_gdn_bad", 3, 2, 128, 128, 8, 2, seed=307)
    sa, ss, unused, snap = _gdn_pair(w)
    slots = _slot_table("cuda", bad=(3, 1000))
    for t in range(w.steps):
        rec = I.gdn_step_inputs(w, t, "cuda")
        oa = sa.new_output()
        sa.step(rec, oa)
        os_ = torch.full((ROWS, w.nheads, w.dv), float("nan"), device="cuda")
        ss.step(_rows(rec), os_, slots=slots)
        torch.cuda.synchronize()
        assert torch.equal(os_[ROW_OF], oa), t
        assert torch.isnan(os_[PAD]).all(), t
    assert H.status(ss) == bd.RSSM_DEV_BAD_SLOT
    _check_state(_gdn_fields(ss), _gdn_fields(sa), unused, snap)


def test_slot_table_is_read_at_replay_time():
    """A graph captured with a slot table serves whatever that table holds when it
    is replayed: the table is device data, read by the kernels."""
    w = W("slots_graph", 3, 4, 64, 128, 2, 8, 1, seed=308)
    sa, ss, A, D, unused, snap = _m2_pair(w, False)
    rec = I.mamba2_step_inputs(w, 0, "cuda")
    rows = _rows(rec)
    slots = torch.full((ROWS,), -1, dtype=torch.int32, device="cuda")  # all padding while capturing
    ys = torch.full((ROWS, w.nheads, w.headdim), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ss.step(rows, A, D, ys, slots=slots)
    torch.cuda.synchronize()
    _check_state(_m2_fields(ss), _m2_fields(sa), unused, snap)  # capture ran nothing
    slots.copy_(_slot_table("cuda"))
    g.replay()
    ya = sa.new_output()
    sa.step(rec, A, D, ya)
    torch.cuda.synchronize()
    assert torch.equal(ys[ROW_OF], ya)
    assert torch.isnan(ys[PAD]).all()
    _check_state(_m2_fields(ss), _m2_fields(sa), unused, snap)
