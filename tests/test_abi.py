"""CPU tests of the C-ABI boundary: the library loads, exports exactly the calls
include/rssm.h declares, and rejects bad arguments on the host before any
launch (no GPU is touched by any of these)."""
import ctypes
import os
import re
import subprocess

import pytest

from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rssm.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return bd.load()


def header_functions():
    text = open(HEADER).read()
    return set(re.findall(r"RSSM_API\s+(?:const\s+)?\w+\*?\s+(rssm_\w+)\s*\(", text))


def test_exports_match_header(lib):
    declared = header_functions()
    assert len(declared) == 28
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == declared
    assert set(bd.EXPORTED) == declared
    for name in declared:
        assert getattr(lib, name) is not None


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "rssm.h"\nint main(void){ rssm_mamba2_desc d; (void)d; return RSSM_OK; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-c", str(src),
                    "-o", str(tmp_path / "t.o")], check=True)


def test_status_strings(lib):
    assert bd.rssm_version() == 200
    for code in (0, -1, -2, -3, -4, 1, 2, 3, 4, 5, 6):
        assert bd.status_string(code) != "unknown status code"
    assert bd.status_string(999) == "unknown status code"


def test_ring_bytes(lib):
    d = bd.mamba2_desc(256, 128, 64, 128, 8, 16)
    assert bd.rssm_mamba2_ring_bytes(d) == [256 * 128 * 16 * 64 * 2] * 2 + [256 * 8 * 16 * 128 * 2] * 2 + [256 * 128 * 16 * 4]
    g = bd.gdn_desc(256, 32, 128, 128, 16)
    assert bd.rssm_gdn_ring_bytes(g) == [256 * 32 * 16 * 128 * 2] * 3 + [256 * 32 * 16 * 4] * 2 + \
        [256 * 32 * 16 * 128 * 4]


ALIGNED = 1 << 20  # a fake, 16-byte aligned address: never dereferenced because validation fails first
ARGS9 = [ALIGNED] * 9  # cursors, x, z, B, C, dt, A, D, y


@pytest.mark.parametrize("desc", [
    (4, 8, 64, 128, 3, 16),    # H % G != 0
    (4, 8, 60, 128, 1, 16),    # headdim not a multiple of 8
    (4, 8, 64, 264, 1, 16),    # dstate > 256
    (4, 8, 64, 128, 1, 0),     # L < 1
    (4, 8, 64, 128, 1, 33),    # L > 32
    (-1, 8, 64, 128, 1, 16),   # negative batch
    (4, 8, 64, 128, 1, 16, 7),  # bad out_dtype
    (4, 8, 64, 128, 1, 16, 0, 9),  # bad read_dtype
    (4, 8, 64, 128, 1, 16, 0, bd.RSSM_FP8_E4M3 + 1),
])
def test_mamba2_desc_validation(lib, desc):
    d = bd.mamba2_desc(*desc)
    ring = bd.rssm_mamba2_ring(*([ALIGNED] * 5))
    assert lib.rssm_mamba2_step(ctypes.byref(d), ALIGNED, None, ctypes.byref(ring), *ARGS9, None, None) == \
        bd.RSSM_ERR_INVALID_ARG


def test_fp8_read_copy_needs_the_specialised_shapes(lib):
    ring = bd.rssm_mamba2_ring(*([ALIGNED] * 5))
    for desc in ((4, 8, 64, 64, 1, 16), (4, 8, 48, 128, 1, 16), (4, 8, 64, 128, 1, 32), (4, 6, 64, 128, 2, 16)):
        d = bd.mamba2_desc(*desc, 0, bd.RSSM_FP8_E4M3)  # dstate != 128, headdim % 64, L > 31, 3 heads per group
        assert lib.rssm_mamba2_step(ctypes.byref(d), ALIGNED, ALIGNED, ctypes.byref(ring), *ARGS9, None, None) == \
            bd.RSSM_ERR_UNSUPPORTED
        assert lib.rssm_mamba2_downcast(ctypes.byref(d), ALIGNED, ALIGNED, None) == bd.RSSM_ERR_UNSUPPORTED
    d = bd.mamba2_desc(4, 8, 64, 128, 1, 16, 0, bd.RSSM_FP8_E4M3)
    assert lib.rssm_mamba2_spec_verify(ctypes.byref(d), 8, ALIGNED, ALIGNED, ctypes.byref(ring), *ARGS9,
                                       None, None) == bd.RSSM_ERR_UNSUPPORTED  # K > 4
    assert lib.rssm_mamba2_downcast(ctypes.byref(d), ALIGNED, ALIGNED + 4, None) == bd.RSSM_ERR_MISALIGNED


def test_empty_batch_is_noop(lib):
    d = bd.mamba2_desc(0, 8, 64, 128, 1, 16)
    assert lib.rssm_mamba2_step(ctypes.byref(d), None, None, None, *([None] * 9), None, None) == bd.RSSM_OK
    assert lib.rssm_mamba2_flush(ctypes.byref(d), None, None, None, None, None, None, None) == bd.RSSM_OK
    assert lib.rssm_mamba2_conventional_step(ctypes.byref(d), *([None] * 9), None) == bd.RSSM_OK


def test_mamba2_pointer_checks(lib):
    d = bd.mamba2_desc(4, 8, 64, 128, 1, 16)
    ring = bd.rssm_mamba2_ring(*([ALIGNED] * 5))
    rb = ctypes.byref(ring)
    assert lib.rssm_mamba2_step(ctypes.byref(d), None, None, rb, *ARGS9, None, None) == bd.RSSM_ERR_INVALID_ARG
    bad = list(ARGS9)
    bad[-1] = ALIGNED + 4  # misaligned y
    assert lib.rssm_mamba2_step(ctypes.byref(d), ALIGNED, None, rb, *bad, None, None) == bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_mamba2_step(ctypes.byref(d), ALIGNED, ALIGNED + 2, rb, *ARGS9, None, None) == bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_mamba2_step(ctypes.byref(d), ALIGNED, None, rb, *ARGS9, ALIGNED + 8, None) == bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_mamba2_step(ctypes.byref(d), ALIGNED, None, None, *ARGS9, None, None) == bd.RSSM_ERR_INVALID_ARG
    ring0 = bd.rssm_mamba2_ring(ALIGNED, ALIGNED, None, ALIGNED, ALIGNED)
    assert lib.rssm_mamba2_step(ctypes.byref(d), ALIGNED, None, ctypes.byref(ring0), *ARGS9, None, None) == \
        bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_mamba2_step(None, ALIGNED, None, rb, *ARGS9, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_mamba2_conventional_step(ctypes.byref(d), ALIGNED, *([ALIGNED] * 7), ALIGNED + 4, None) == \
        bd.RSSM_ERR_MISALIGNED


def test_verify_n_new_range(lib):
    d = bd.mamba2_desc(4, 8, 64, 128, 1, 16)
    ring = bd.rssm_mamba2_ring(*([ALIGNED] * 5))
    for n_new in (0, 17, -1):
        rc = lib.rssm_mamba2_spec_verify(ctypes.byref(d), n_new, ALIGNED, None, ctypes.byref(ring), *ARGS9,
                                         None, None)
        assert rc == bd.RSSM_ERR_INVALID_ARG


def test_cursor_call_validation(lib):
    assert lib.rssm_commit_cursors(ALIGNED, ALIGNED, 4, 0, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_commit_cursors(ALIGNED, ALIGNED, 4, 33, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_commit_cursors(ALIGNED, None, 4, 16, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_commit_cursors(ALIGNED + 4, ALIGNED, 4, 16, None, None) == bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_commit_cursors(None, None, 0, 16, None, None) == bd.RSSM_OK
    assert lib.rssm_reset_cursors(None, None, 0, 4, None, None) == bd.RSSM_OK
    assert lib.rssm_reset_cursors(ALIGNED, None, 2, 4, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_reset_cursors(ALIGNED, ALIGNED, -1, 4, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_checkpoint_downcast(None, None, 0, bd.RSSM_BF16, None) == bd.RSSM_OK
    assert lib.rssm_checkpoint_downcast(ALIGNED, ALIGNED + 2, 8, bd.RSSM_F16, None) == bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_checkpoint_downcast(ALIGNED, ALIGNED, 8, bd.RSSM_F32, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_selftest_bounded_wait(None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_selftest_bounded_wait(ALIGNED + 4, None) == bd.RSSM_ERR_MISALIGNED


def test_gdn_validation(lib):
    ring = bd.rssm_gdn_ring(*([ALIGNED] * 6))
    for desc in ((4, 2, 60, 128, 16), (4, 2, 128, 512, 16), (4, 0, 128, 128, 16), (4, 2, 128, 128, 40)):
        d = bd.gdn_desc(*desc)
        assert lib.rssm_gdn_step(ctypes.byref(d), ALIGNED, ctypes.byref(ring), *([ALIGNED] * 7), None, None) == \
            bd.RSSM_ERR_INVALID_ARG
    d = bd.gdn_desc(4, 2, 128, 128, 16)
    assert lib.rssm_gdn_step(ctypes.byref(d), ALIGNED + 4, ctypes.byref(ring), *([ALIGNED] * 7), None, None) == \
        bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_gdn_flush(ctypes.byref(d), ALIGNED, None, ALIGNED, None, None) == bd.RSSM_ERR_INVALID_ARG
    d0 = bd.gdn_desc(0, 2, 128, 128, 16)
    assert lib.rssm_gdn_flush(ctypes.byref(d0), None, None, None, None, None) == bd.RSSM_OK
    # the step and the prime need the ring's e field
    no_e = bd.rssm_gdn_ring(*([ALIGNED] * 5), None)
    assert lib.rssm_gdn_step(ctypes.byref(d), ALIGNED, ctypes.byref(no_e), *([ALIGNED] * 7), None, None) == \
        bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_gdn_prime(ctypes.byref(d), ALIGNED, ctypes.byref(no_e), ALIGNED, None, None) == \
        bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_gdn_prime(ctypes.byref(d), ALIGNED, None, ALIGNED, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_gdn_prime(ctypes.byref(d0), None, None, None, None, None) == bd.RSSM_OK


def test_state_slot_host_checks(lib):
    """State slots: ring sizes follow n_slots; calls outside the shape-specialised
    decode kernels reject a slot table; n_slots is range-checked. Every case
    returns before any launch."""
    d = bd.mamba2_desc(4, 8, 64, 128, 1, 16, state_slots=ALIGNED, n_slots=10)
    assert bd.rssm_mamba2_ring_bytes(d)[0] == 10 * 8 * 16 * 64 * 2
    g = bd.gdn_desc(4, 2, 128, 128, 16, state_slots=ALIGNED, n_slots=7)
    assert bd.rssm_gdn_ring_bytes(g)[5] == 7 * 2 * 16 * 128 * 4
    ring = bd.rssm_mamba2_ring(*([ALIGNED] * 5))
    rb = ctypes.byref(ring)
    generic = bd.mamba2_desc(4, 8, 48, 64, 1, 16, state_slots=ALIGNED, n_slots=8)  # not dstate 128
    assert lib.rssm_mamba2_step(ctypes.byref(generic), ALIGNED, None, rb, *ARGS9, None, None) == \
        bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_mamba2_spec_verify(ctypes.byref(generic), 2, ALIGNED, None, rb, *ARGS9, None, None) == \
        bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_mamba2_spec_verify(ctypes.byref(d), 8, ALIGNED, None, rb, *ARGS9, None, None) == \
        bd.RSSM_ERR_UNSUPPORTED  # K > 4: the persistent verify takes no slot table
    assert lib.rssm_mamba2_flush(ctypes.byref(d), ALIGNED, None, rb, ALIGNED, ALIGNED, None, None) == \
        bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_mamba2_conventional_step(ctypes.byref(d), *([ALIGNED] * 9), None) == bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_mamba2_downcast(ctypes.byref(d), ALIGNED, ALIGNED, None) == bd.RSSM_ERR_UNSUPPORTED
    for n_slots, rc in ((-1, bd.RSSM_ERR_INVALID_ARG), (70000, bd.RSSM_ERR_UNSUPPORTED)):
        bad = bd.mamba2_desc(4, 8, 64, 128, 1, 16, state_slots=ALIGNED, n_slots=n_slots)
        assert lib.rssm_mamba2_step(ctypes.byref(bad), ALIGNED, None, rb, *ARGS9, None, None) == rc
        badg = bd.gdn_desc(4, 2, 128, 128, 16, state_slots=ALIGNED, n_slots=n_slots)
        assert lib.rssm_gdn_flush(ctypes.byref(badg), ALIGNED, None, ALIGNED, None, None) == rc
    gring = bd.rssm_gdn_ring(*([ALIGNED] * 6))
    g64 = bd.gdn_desc(4, 2, 64, 128, 16, state_slots=ALIGNED, n_slots=8)  # not dk = dv = 128
    assert lib.rssm_gdn_step(ctypes.byref(g64), ALIGNED, ctypes.byref(gring), *([ALIGNED] * 7), None, None) == \
        bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_gdn_spec_verify(ctypes.byref(g64), 2, ALIGNED, ctypes.byref(gring), *([ALIGNED] * 7), None,
                                    None) == bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_gdn_flush(ctypes.byref(g), ALIGNED, ctypes.byref(gring), ALIGNED, None, None) == \
        bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_gdn_prime(ctypes.byref(g), ALIGNED, ctypes.byref(gring), ALIGNED, None, None) == \
        bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_gdn_conventional_step(ctypes.byref(g), *([ALIGNED] * 8), None) == bd.RSSM_ERR_UNSUPPORTED
    # commit with slots
    assert lib.rssm_commit_cursors_slots(ALIGNED, ALIGNED, None, 4, 8, 16, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_commit_cursors_slots(ALIGNED, ALIGNED, ALIGNED, 4, -1, 16, None, None) == \
        bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_commit_cursors_slots(ALIGNED, ALIGNED, ALIGNED, 4, 8, 0, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_commit_cursors_slots(None, None, None, 0, 8, 16, None, None) == bd.RSSM_OK


def test_kda_host_checks(lib):
    """Kimi Delta Attention: ring sizes (g one fp32 per key channel), the replay
    calls' shape limits and their argument checks; every case returns before a launch."""
    d = bd.kda_desc(4, 2, 128, 128, 16)
    assert bd.rssm_kda_ring_bytes(d) == [4 * 2 * 16 * 128 * 2] * 3 + [4 * 2 * 16 * 128 * 4, 4 * 2 * 16 * 4,
                                                                       4 * 2 * 16 * 128 * 4]
    ring = bd.rssm_kda_ring(*([ALIGNED] * 6))
    rb = ctypes.byref(ring)
    for desc in ((4, 2, 64, 128, 16), (4, 2, 128, 64, 16), (4, 2, 128, 128, 32)):  # dk, dv != 128; L = 32
        dd = bd.kda_desc(*desc)
        assert lib.rssm_kda_step(ctypes.byref(dd), ALIGNED, rb, *([ALIGNED] * 7), None, None) == \
            bd.RSSM_ERR_UNSUPPORTED
    dd = bd.kda_desc(4, 2, 64, 128, 16)
    assert lib.rssm_kda_flush(ctypes.byref(dd), ALIGNED, rb, ALIGNED, None, None) == bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_kda_prime(ctypes.byref(dd), ALIGNED, rb, ALIGNED, None, None) == bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_kda_step(ctypes.byref(d), ALIGNED + 4, rb, *([ALIGNED] * 7), None, None) == \
        bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_kda_step(ctypes.byref(d), ALIGNED, None, *([ALIGNED] * 7), None, None) == bd.RSSM_ERR_INVALID_ARG
    no_g = bd.rssm_kda_ring(ALIGNED, ALIGNED, ALIGNED, None, ALIGNED, ALIGNED)
    assert lib.rssm_kda_flush(ctypes.byref(d), ALIGNED, ctypes.byref(no_g), ALIGNED, None, None) == \
        bd.RSSM_ERR_INVALID_ARG
    ds = bd.kda_desc(4, 2, 128, 128, 16, state_slots=ALIGNED, n_slots=8)
    assert lib.rssm_kda_flush(ctypes.byref(ds), ALIGNED, rb, ALIGNED, None, None) == bd.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_kda_conventional_step(ctypes.byref(ds), *([ALIGNED] * 8), None) == bd.RSSM_ERR_UNSUPPORTED
    d0 = bd.kda_desc(0, 2, 128, 128, 16)
    assert lib.rssm_kda_step(ctypes.byref(d0), None, None, *([None] * 7), None, None) == bd.RSSM_OK
    # the speculative verify: n_new in [1, L]; K <= 4, L + K <= 32 and dk = dv = 128 on its kernel (with or
    # without state slots)
    args = (ALIGNED, rb, *([ALIGNED] * 8))
    for n_new in (0, 17, -1):
        assert lib.rssm_kda_spec_verify(ctypes.byref(d), n_new, *args, None, None) == bd.RSSM_ERR_INVALID_ARG
    assert lib.rssm_kda_spec_verify(ctypes.byref(d), 5, *args, None, None) == bd.RSSM_ERR_UNSUPPORTED
    d30 = bd.kda_desc(4, 2, 128, 128, 30)
    assert lib.rssm_kda_spec_verify(ctypes.byref(d30), 3, *args, None, None) == bd.RSSM_ERR_UNSUPPORTED
    d64 = bd.kda_desc(4, 2, 64, 128, 16)
    assert lib.rssm_kda_spec_verify(ctypes.byref(d64), 4, *args, None, None) == bd.RSSM_ERR_UNSUPPORTED
    ds64 = bd.kda_desc(4, 2, 64, 128, 16, state_slots=ALIGNED, n_slots=8)
    assert lib.rssm_kda_spec_verify(ctypes.byref(ds64), 4, *args, None, None) == bd.RSSM_ERR_UNSUPPORTED
    bad = (ALIGNED, rb, *([ALIGNED] * 7), ALIGNED + 4)  # misaligned o
    assert lib.rssm_kda_spec_verify(ctypes.byref(d), 4, *bad, None, None) == bd.RSSM_ERR_MISALIGNED
    assert lib.rssm_kda_spec_verify(ctypes.byref(d0), 4, *([None] * 10), None, None) == bd.RSSM_OK
    assert lib.rssm_kda_conventional_step(ctypes.byref(bd.kda_desc(4, 2, 60, 128, 16)), *([ALIGNED] * 8), None) == \
        bd.RSSM_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(bd, "_lib", None)
    monkeypatch.setattr(bd, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        bd.load()


def test_slot_tables_are_checked_before_any_call():
    """The state layer refuses a slot table the kernels would misread (not
    int32, not on the state's device, not contiguous); nothing is launched."""
    import torch

    from recurrent_state_decode_gb300.state import GDNState, Mamba2State
    m = Mamba2State(2, 4, 64, 128, 2, 8, device="cpu")
    g = GDNState(2, 2, 128, 128, 8, device="cpu")
    for st in (m, g):
        with pytest.raises(ValueError):
            st.slot_desc(torch.zeros(3, dtype=torch.int64))
        with pytest.raises(ValueError):
            st.slot_desc(torch.zeros(6, dtype=torch.int32)[::2])
        d = st.slot_desc(torch.tensor([1, -1, 0], dtype=torch.int32))
        assert d.batch == 3 and d.n_slots == 2
    with pytest.raises(ValueError):
        m.commit(torch.zeros(3, dtype=torch.int32), slots=torch.zeros(3, dtype=torch.int64))


def test_record_tensors_are_checked_before_any_call():
    """The state layer refuses record, output and kept tensors the kernels
    would misread: a wrong dtype, device, row count or shape, or a
    non-contiguous view raises ValueError before the C ABI is reached."""
    import torch

    from recurrent_state_decode_gb300.state import GDNState, KDAState, Mamba2State
    m = Mamba2State(2, 4, 64, 128, 2, 8, device="cpu")
    bf, f32 = torch.bfloat16, torch.float32
    rec = {"x": torch.zeros(2, 4, 64, dtype=bf), "z": torch.zeros(2, 4, 64, dtype=bf),
           "B": torch.zeros(2, 2, 128, dtype=bf), "C": torch.zeros(2, 2, 128, dtype=bf),
           "dt": torch.zeros(2, 4, dtype=f32)}
    A, D, y = torch.zeros(4), torch.zeros(4), torch.zeros(2, 4, 64)
    bad = [dict(rec, dt=torch.zeros(2, 4, dtype=bf)),                      # dt not fp32
           dict(rec, x=torch.zeros(2, 4, 128, dtype=bf)[..., ::2]),        # a strided view of x
           dict(rec, B=torch.zeros(1, 2, 128, dtype=bf)),                  # too few rows
           dict(rec, C=torch.zeros(2, 2, 64, dtype=bf)),                   # wrong dstate
           {k: v for k, v in rec.items() if k != "z"}]                     # a missing field
    if torch.cuda.is_available():
        bad.append(dict(rec, x=rec["x"].cuda()))                           # another device
    for r in bad:
        with pytest.raises(ValueError):
            m.step(r, A, D, y)
    with pytest.raises(ValueError):
        m.step(rec, A, D, torch.zeros(2, 4, 64, dtype=bf))                 # y of the wrong dtype
    with pytest.raises(ValueError):
        m.step(rec, A.double(), D, y)                                      # A not fp32
    with pytest.raises(ValueError):
        m.step(rec, A, D, y, slots=torch.tensor([1, -1, 0], dtype=torch.int32))  # 2 record rows for 3 slot rows
    vrec = {k: torch.stack([v, v], 1) for k, v in rec.items()}
    with pytest.raises(ValueError):
        m.verify(vrec, A, D, torch.zeros(2, 3, 4, 64))                     # y with 3 drafts for 2
    with pytest.raises(ValueError):
        m.verify(rec, A, D, y)                                             # no draft axis
    with pytest.raises(ValueError):
        m.commit(torch.zeros(2, dtype=torch.int64))                        # kept not int32
    with pytest.raises(ValueError):
        m.commit(torch.zeros(3, dtype=torch.int32))                        # kept of the wrong length
    with pytest.raises(ValueError):
        m.flush(torch.zeros(3))
    g = GDNState(2, 2, 128, 128, 8, device="cpu")
    grec = {"q": torch.zeros(2, 2, 128, dtype=bf), "k": torch.zeros(2, 2, 128, dtype=bf),
            "v": torch.zeros(2, 2, 128, dtype=bf), "g": torch.zeros(2, 2), "beta": torch.zeros(2, 2)}
    with pytest.raises(ValueError):
        g.step(dict(grec, v=torch.zeros(2, 2, 64, dtype=bf)), torch.zeros(2, 2, 128))
    with pytest.raises(ValueError):
        g.step(grec, torch.zeros(2, 2, 128, dtype=bf))                     # o of the wrong dtype
    k = KDAState(2, 2, 128, 128, 8, device="cpu")
    with pytest.raises(ValueError):
        k.step(grec, torch.zeros(2, 2, 128))                               # KDA g is per key channel
    with pytest.raises(ValueError):
        k.verify({f: torch.stack([v, v], 1) for f, v in grec.items()}, torch.zeros(2, 2, 2, 128))


def test_emulated_step_host_checks(lib):
    """rssm_mamba2_step_emulated: the workspace size query, the format / scale
    pairs it takes, the shapes and the workspace size it needs."""
    d = bd.mamba2_desc(4, 8, 64, 128, 2, 16)
    n = bd.rssm_mamba2_emulated_workspace_bytes(d)
    assert n == 4 * 8 * 1 * 8                # one (error, norm) fp32 pair per block (sequence, head, 64 rows)
    ring = bd.rssm_mamba2_ring(*([ALIGNED] * 5))
    args = [ALIGNED] * 9                     # x, z, B, C, dt, A, D, y, err

    def call(desc, emu, nbytes=n, ws=ALIGNED):
        return lib.rssm_mamba2_step_emulated(ctypes.byref(desc), None if emu is None else ctypes.byref(emu), ALIGNED,
                                             ctypes.byref(ring), ALIGNED, *args[:8], args[8], ws, nbytes, None, None)
    ok = [(bd.RSSM_EMU_BF16, 0), (bd.RSSM_EMU_F16, 0), (bd.RSSM_EMU_E4M3, 1), (bd.RSSM_EMU_E5M2, 2),
          (bd.RSSM_EMU_INT8, 1), (bd.RSSM_EMU_INT8, 2)]
    bad = [(bd.RSSM_EMU_BF16, 1), (bd.RSSM_EMU_F16, 2), (bd.RSSM_EMU_E4M3, 0), (bd.RSSM_EMU_INT8, 0), (0, 0),
           (6, 1), (bd.RSSM_EMU_E4M3, 3)]
    for f, sc in bad:
        assert call(d, bd.emulation(f, sc)) == bd.RSSM_ERR_INVALID_ARG, (f, sc)
    assert call(d, None) == bd.RSSM_ERR_INVALID_ARG
    for f, sc in ok:   # valid pairs pass every host check; an empty batch launches nothing
        assert call(bd.mamba2_desc(0, 8, 64, 128, 2, 16), bd.emulation(f, sc)) == bd.RSSM_OK
    emu = bd.emulation(bd.RSSM_EMU_E4M3, bd.RSSM_EMU_SCALE_ROW)
    assert call(d, emu, nbytes=n - 1) == bd.RSSM_ERR_INVALID_ARG
    assert call(d, emu, ws=None) == bd.RSSM_ERR_INVALID_ARG
    assert call(d, emu, ws=ALIGNED + 8) == bd.RSSM_ERR_MISALIGNED
    for shape in ((4, 8, 64, 64, 2, 16), (4, 8, 48, 128, 2, 16), (4, 8, 64, 128, 2, 32), (4, 6, 64, 128, 2, 16)):
        ds = bd.mamba2_desc(*shape)
        assert call(ds, emu) == bd.RSSM_ERR_UNSUPPORTED, shape
        with pytest.raises(bd.RssmError):
            bd.rssm_mamba2_emulated_workspace_bytes(ds)
    slots = bd.mamba2_desc(4, 8, 64, 128, 2, 16, state_slots=ALIGNED, n_slots=4)
    assert call(slots, emu) == bd.RSSM_ERR_UNSUPPORTED


def test_noalloc_step_host_checks(lib):
    """The no-allocation emulated step takes the emulated step's checks, and a
    launch beyond its static scratch (more than RSSM_NOALLOC_MAX_WARPS warps)
    is refused on the host with RSSM_ERR_UNSUPPORTED."""
    ring = bd.rssm_mamba2_ring(*([ALIGNED] * 5))
    emu = bd.emulation(bd.RSSM_EMU_E4M3, bd.RSSM_EMU_SCALE_TILE64)

    def call(desc, e=emu):
        return lib.rssm_mamba2_step_emulated_noalloc(ctypes.byref(desc), ctypes.byref(e), ALIGNED, ctypes.byref(ring),
                                                     *([ALIGNED] * 10), None, None)
    assert bd.RSSM_NOALLOC_MAX_WARPS == 262144
    big = bd.mamba2_desc(513, 128, 64, 128, 8, 16)          # 513 * 128 * 4 warps > 262144
    assert call(big) == bd.RSSM_ERR_UNSUPPORTED
    assert call(bd.mamba2_desc(4, 8, 64, 128, 2, 16), bd.emulation(bd.RSSM_EMU_E4M3, 0)) == bd.RSSM_ERR_INVALID_ARG
    assert call(bd.mamba2_desc(4, 8, 64, 64, 2, 16)) == bd.RSSM_ERR_UNSUPPORTED
    assert call(bd.mamba2_desc(0, 8, 64, 128, 2, 16)) == bd.RSSM_OK
