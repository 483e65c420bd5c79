"""The kernels' bounded waits: a wait that runs out reports RSSM_DEV_TIMEOUT to
the device status word and returns, and the context stays usable. The wait is
made to run out on an mbarrier armed for bytes that no copy delivers; nothing
faults and nothing hangs."""
import pytest
import torch

import harness as H
from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.inputs import Mamba2Workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from recurrent_state_decode_gb300 import build
    build.build()
    bd.load()


def test_expired_wait_reports_timeout_and_the_context_stays_usable():
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert bd.rssm_selftest_bounded_wait(status) == bd.RSSM_OK
    torch.cuda.synchronize()
    assert int(status[0]) == bd.RSSM_DEV_TIMEOUT
    # a decode step afterwards runs normally
    w = W("after_timeout", 2, 4, 64, 128, 2, 8, 1, seed=501)
    st, A, D, _, _, _ = H.mamba2_setup(w, "cuda")
    y = st.new_output()
    st.step(I.mamba2_step_inputs(w, 0, "cuda"), A, D, y)
    torch.cuda.synchronize()
    assert H.status(st) == 0
    assert torch.isfinite(y).all()


def test_selftest_argument_checks():
    assert bd.rssm_selftest_bounded_wait(None) == bd.RSSM_ERR_INVALID_ARG
