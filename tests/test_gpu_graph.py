"""Every call is asynchronous, allocates nothing and never synchronises, so a
sequence of calls can be captured into a CUDA graph and replayed: the replay
must reproduce an eager run bit for bit (outputs, checkpoints, rings, cursors)."""
import pytest
import torch

import harness as H
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import GDNWorkload as GW
from recurrent_state_decode_gb300.inputs import Mamba2Workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def _capture(fn):
    """Run fn() under CUDA-graph capture on a side stream, then replay it once."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    g.replay()
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", [W("graph_fast", 3, 4, 64, 128, 2, 8, 12, seed=201),       # shape-specialised kernels
                               W("graph_generic", 3, 6, 24, 40, 3, 5, 12, seed=202)],    # generic kernels
                         ids=lambda w: w.name)
def test_mamba2_steps_replay_from_a_graph(w):
    dev = "cuda"
    recs = [I.mamba2_step_inputs(w, t, dev) for t in range(w.steps)]
    sa, A, D, _, _, _ = H.mamba2_setup(w, dev)
    sb, _, _, _, _, _ = H.mamba2_setup(w, dev)
    ya = [sa.new_output() for _ in range(w.steps)]
    yb = [sb.new_output() for _ in range(w.steps)]
    for t in range(w.steps):
        sa.step(recs[t], A, D, ya[t])
    torch.cuda.synchronize()

    def steps():
        for t in range(w.steps):
            sb.step(recs[t], A, D, yb[t])

    _capture(steps)
    for t in range(w.steps):
        assert torch.equal(ya[t], yb[t]), t
    for fa, fb in ((sa.ckpt, sb.ckpt), (sa.rx, sb.rx), (sa.rB, sb.rB), (sa.rdt, sb.rdt), (sa.cursors, sb.cursors)):
        assert torch.equal(fa, fb)
    assert H.status(sa) == 0 and H.status(sb) == 0


def test_mamba2_verify_commit_replay_from_a_graph():
    w = W("graph_spec", 3, 4, 64, 128, 2, 8, 6, seed=203, drafts=3)
    dev = "cuda"
    recs = [I.mamba2_verify_inputs(w, t, dev) for t in range(w.steps)]
    kepts = [I.accepted_kept(w, t, dev) for t in range(w.steps)]
    sa, A, D, _, _, _ = H.mamba2_setup(w, dev)
    sb, _, _, _, _, _ = H.mamba2_setup(w, dev)
    ya = [sa.new_output(w.n_new) for _ in range(w.steps)]
    yb = [sb.new_output(w.n_new) for _ in range(w.steps)]
    for t in range(w.steps):
        sa.verify(recs[t], A, D, ya[t])
        sa.commit(kepts[t])
    torch.cuda.synchronize()

    def spec():
        for t in range(w.steps):
            sb.verify(recs[t], A, D, yb[t])
            sb.commit(kepts[t])

    _capture(spec)
    for t in range(w.steps):
        assert torch.equal(ya[t], yb[t]), t
    assert torch.equal(sa.ckpt, sb.ckpt) and torch.equal(sa.cursors, sb.cursors)
    assert H.status(sa) == 0 and H.status(sb) == 0


def test_gdn_steps_replay_from_a_graph():
    w = GW("graph_gdn", 2, 2, 128, 128, 8, 12, seed=204)
    dev = "cuda"
    recs = [I.gdn_step_inputs(w, t, dev) for t in range(w.steps)]
    sa, _, _, _ = H.gdn_setup(w, dev)
    sb, _, _, _ = H.gdn_setup(w, dev)
    oa = [sa.new_output() for _ in range(w.steps)]
    ob = [sb.new_output() for _ in range(w.steps)]
    for t in range(w.steps):
        sa.step(recs[t], oa[t])
    torch.cuda.synchronize()

    def steps():
        for t in range(w.steps):
            sb.step(recs[t], ob[t])

    _capture(steps)
    for t in range(w.steps):
        assert torch.equal(oa[t], ob[t]), t
    assert torch.equal(sa.S, sb.S) and torch.equal(sa.re, sb.re) and torch.equal(sa.cursors, sb.cursors)
    assert H.status(sa) == 0 and H.status(sb) == 0


def test_kda_steps_replay_from_a_graph():
    from recurrent_state_decode_gb300.inputs import KDAWorkload as KW
    from recurrent_state_decode_gb300.state import kda_from_workload
    w = KW("graph_kda", 2, 2, 128, 128, 8, 12, seed=205)
    dev = "cuda"
    recs = [I.kda_step_inputs(w, t, dev) for t in range(w.steps)]
    sa, _, _, _ = kda_from_workload(w, dev)
    sb, _, _, _ = kda_from_workload(w, dev)
    oa = [sa.new_output() for _ in range(w.steps)]
    ob = [sb.new_output() for _ in range(w.steps)]
    for t in range(w.steps):
        sa.step(recs[t], oa[t])
    torch.cuda.synchronize()

    def steps():
        for t in range(w.steps):
            sb.step(recs[t], ob[t])

    _capture(steps)
    for t in range(w.steps):
        assert torch.equal(oa[t], ob[t]), t
    for fa, fb in ((sa.S, sb.S), (sa.rg, sb.rg), (sa.re, sb.re), (sa.rk, sb.rk), (sa.cursors, sb.cursors)):
        assert torch.equal(fa, fb)
    assert H.status(sa) == 0 and H.status(sb) == 0


@pytest.mark.parametrize("kda", [False, True], ids=["gdn", "kda"])
def test_delta_verify_commit_replay_from_a_graph(kda):
    """Speculative verifies and commits of the delta-rule layers, eager against
    replayed from a graph, with state slots on the replayed side (a permuted
    batch: the table is device data, read when the graph runs)."""
    from recurrent_state_decode_gb300.inputs import KDAWorkload as KW
    from recurrent_state_decode_gb300.state import GDNState, KDAState, gdn_from_workload, kda_from_workload
    dev = "cuda"
    if kda:
        w = KW("graph_kda_spec", 3, 2, 128, 128, 8, 6, seed=206, drafts=3)
        make, inputs, cls = kda_from_workload, I.kda_verify_inputs, KDAState
    else:
        w = GW("graph_gdn_spec", 3, 2, 128, 128, 8, 6, seed=207, drafts=3)
        make, inputs, cls = gdn_from_workload, I.gdn_verify_inputs, GDNState
    recs = [inputs(w, t, dev) for t in range(w.steps)]
    kepts = [I.accepted_kept(w, t, dev) for t in range(w.steps)]
    sa = make(w, dev)[0]
    sb = cls(w.batch, w.nheads, w.dk, w.dv, w.buf_len, dev)
    perm = torch.tensor([2, 0, 1], dtype=torch.int32, device=dev)  # batch row b uses state row perm[b]
    fields = ("S", "rq", "rk", "rv", "rg", "rbeta", "re", "cursors")
    for f in fields:
        getattr(sb, f)[perm.long()] = getattr(sa, f)
    oa = [sa.new_verify_output(w.n_new) for _ in range(w.steps)]
    ob = [sb.new_verify_output(w.n_new) for _ in range(w.steps)]
    for t in range(w.steps):
        sa.verify(recs[t], oa[t])
        sa.commit(kepts[t])
    torch.cuda.synchronize()

    def spec():
        for t in range(w.steps):
            sb.verify(recs[t], ob[t], slots=perm)
            sb.commit(kepts[t], slots=perm)

    _capture(spec)
    for t in range(w.steps):
        assert torch.equal(oa[t], ob[t]), t
    for f in fields:
        assert torch.equal(getattr(sb, f)[perm.long()], getattr(sa, f)), f
    assert H.status(sa) == 0 and H.status(sb) == 0
