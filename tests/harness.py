"""Shared helpers for the parity tests: set up a decode session on the GPU
from a seeded workload, feed the same records to the oracle, compare."""
import numpy as np
import torch

from recurrent_state_decode_gb300 import binding as bd
from recurrent_state_decode_gb300 import inputs as I
from recurrent_state_decode_gb300.state import gdn_from_workload, mamba2_from_workload

F64 = I.to_f64


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def half_ulp_bf16(v):
    """Half a bf16 unit in the last place of |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def bf16_excess(y_gpu, y_ref):
    """max_i(|y_gpu - y_ref| - half_ulp_bf16(y_ref)) / RMS(y_ref): the bf16-output
    check (output rounding alone may cost half an ulp; the rest must stay
    below 2e-3 of the output RMS)."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    return float(np.max(np.abs(y_gpu - y_ref) - half_ulp_bf16(y_ref)) / rms)


class Feed:
    """Lets a lock-step loop hand each record to an oracle session generator."""

    def __init__(self):
        self.rec = None

    def __iter__(self):
        while True:
            yield self.rec


def sub(rec, seqs):
    return {k: F64(v[seqs]) for k, v in rec.items()}


def mamba2_setup(w, device="cuda", out_dtype=bd.RSSM_F32, read_copy=None):
    """GPU session at the start of workload w: checkpoint, pre-filled window, cursors."""
    return mamba2_from_workload(w, device, out_dtype, read_copy)


def gdn_setup(w, device="cuda", out_dtype=bd.RSSM_F32):
    return gdn_from_workload(w, device, out_dtype)


def status(st):
    return int(st.status.item())


def bits16(t):
    """The 16-bit codes of a bf16 / fp16 tensor, as uint16 numpy."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_read_copy(st, b):
    """State row b's read copy equals the oracle's rounding of its fp32
    checkpoint bit for bit (bf16 / fp16 codes; e4m3 codes and row scales)."""
    from oracle import readcopy as rc
    ck = st.ckpt[b].cpu().numpy()
    if getattr(st, "read_q", None) is not None:
        q, sc = rc.e4m3_rows(ck)
        np.testing.assert_array_equal(st.read_q[b].cpu().numpy(), q)
        np.testing.assert_array_equal(st.read_scale[b].cpu().numpy(), sc)
    elif st.ckpt_read.dtype == torch.float16:
        np.testing.assert_array_equal(bits16(st.ckpt_read[b]), rc.fp16_bits(rc.to_fp16(ck)))
    else:
        np.testing.assert_array_equal(bits16(st.ckpt_read[b]), rc.bf16_bits(rc.to_bf16(ck)))
