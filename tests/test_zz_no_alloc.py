"""rssm_mamba2_step_emulated_noalloc: the emulated-precision decode step for
callers that cannot allocate device memory while they decode -- a host that
has already reserved the GPU's memory for its own pools, or that hands the
library a stream but no allocator. It keeps its scratch (the per-block error
sums) in a static device array inside the library instead of a workspace
argument.

Two calls in a row through the C ABI, each against rssm_mamba2_step_emulated
given a workspace, on identical states: outputs within the fp32-path
tolerance (1e-4 relative L2), error reports within 1e-5 relative, checkpoints
within 1e-5 relative L2 and cursors equal. The two calls use different
formats, so a sum left in the shared array by the first call would show in
the second's report. This file is collected last and needs no other test.
"""
import numpy as np
import pytest
import torch

from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import Mamba2Workload as W
from recurrent_state_decode_gb300.state import mamba2_from_workload

pytestmark = pytest.mark.gpu

TOL_Y32, TOL_CKPT, TOL_ERR = 1e-4, 1e-5, 1e-5


def rel_l2(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def test_noalloc_step_matches_the_workspace_step_twice():
    dev = "cuda"
    # L = 4 from staggered windows: the two calls include flushing sequences
    w = W("noalloc", 3, 8, 128, 128, 2, 4, 2, seed=701)
    sa, A, D, _, _, _ = mamba2_from_workload(w, dev, bd.RSSM_F32, read_copy=False)
    sb, _, _, _, _, _ = mamba2_from_workload(w, dev, bd.RSSM_F32, read_copy=False)
    nbytes = bd.rssm_mamba2_emulated_workspace_bytes(sa.desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    err_a = torch.zeros(2, dtype=torch.float64, device=dev)
    err_b = torch.zeros(2, dtype=torch.float64, device=dev)
    formats = [bd.emulation(bd.RSSM_EMU_E4M3, bd.RSSM_EMU_SCALE_TILE64),
               bd.emulation(bd.RSSM_EMU_INT8, bd.RSSM_EMU_SCALE_ROW)]
    flushed = 0
    for t, emu in enumerate(formats):
        rec = I.mamba2_step_inputs(w, t, dev)
        counts = sa.cursors[:, 1].clone()
        ya, yb = sa.new_output(), sb.new_output()
        args = (rec["x"], rec["z"], rec["B"], rec["C"], rec["dt"], A, D)
        bd.check(bd.rssm_mamba2_step_emulated(sa.desc, emu, sa.ckpt, sa.ring, sa.cursors, *args, ya, err_a, ws,
                                              nbytes, sa.status), "rssm_mamba2_step_emulated")
        bd.check(bd.rssm_mamba2_step_emulated_noalloc(sb.desc, emu, sb.ckpt, sb.ring, sb.cursors, *args, yb, err_b,
                                                      sb.status), "rssm_mamba2_step_emulated_noalloc")
        torch.cuda.synchronize()
        flushed += int((counts + 1 == w.buf_len).sum())
        assert rel_l2(yb, ya) <= TOL_Y32, t
        ea, na = err_a.tolist()
        eb, nb = err_b.tolist()
        assert ea > 0 and na > 0
        assert eb == pytest.approx(ea, rel=TOL_ERR) and nb == pytest.approx(na, rel=TOL_ERR), t
        assert rel_l2(sb.ckpt, sa.ckpt) <= TOL_CKPT, t
        assert torch.equal(sb.cursors, sa.cursors), t
    assert flushed > 0
    assert int(sa.status.item()) == 0 and int(sb.status.item()) == 0
