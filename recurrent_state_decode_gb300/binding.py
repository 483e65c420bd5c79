"""ctypes binding of librssm: the C-ABI calls under their own names.

Argument marshalling only. A tensor argument may be a torch tensor (its
``data_ptr()`` is passed), a raw integer address, or ``None`` (NULL). Streams
default to torch's current stream on the tensors' device. Every function
returns the library's integer status; ``check`` raises on a negative one.
Loading fails loudly when the library has not been built: there is no
fallback path.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "librssm.so")

RSSM_OK = 0
RSSM_ERR_INVALID_ARG = -1
RSSM_ERR_UNSUPPORTED = -2
RSSM_ERR_MISALIGNED = -3
RSSM_ERR_CUDA = -4
RSSM_DEV_OK = 0
RSSM_DEV_BAD_CURSOR = 1
RSSM_DEV_WINDOW_FULL = 2
RSSM_DEV_PENDING = 3
RSSM_DEV_BAD_KEPT = 4
RSSM_DEV_BAD_SLOT = 5
RSSM_DEV_TIMEOUT = 6
RSSM_F32 = 0
RSSM_BF16 = 1
RSSM_F16 = 2
RSSM_FP8_E4M3 = 3
RSSM_EMU_BF16 = 1
RSSM_EMU_F16 = 2
RSSM_EMU_E4M3 = 3
RSSM_EMU_E5M2 = 4
RSSM_EMU_INT8 = 5
RSSM_EMU_SCALE_NONE = 0
RSSM_EMU_SCALE_ROW = 1
RSSM_EMU_SCALE_TILE64 = 2

c_int, c_size_t, c_void_p, c_char_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p


class rssm_mamba2_desc(ctypes.Structure):
    _fields_ = [(n, c_int) for n in ("batch", "nheads", "headdim", "dstate", "ngroups", "buf_len", "out_dtype",
                                     "read_dtype")] + [("state_slots", c_void_p), ("n_slots", c_int)]


class rssm_mamba2_ring(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("x", "z", "B", "C", "dt")]


class rssm_gdn_desc(ctypes.Structure):
    _fields_ = [(n, c_int) for n in ("batch", "nheads", "dk", "dv", "buf_len", "out_dtype")] + [
        ("state_slots", c_void_p), ("n_slots", c_int)]


class rssm_gdn_ring(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("q", "k", "v", "g", "beta", "e")]


class rssm_emulation(ctypes.Structure):
    _fields_ = [("format", c_int), ("scale", c_int)]


rssm_kda_desc = rssm_gdn_desc   # the same struct in rssm.h
rssm_kda_ring = rssm_gdn_ring   # same fields; g holds one log decay per key channel


P = c_void_p
_SIGNATURES = {
    "rssm_version": (c_int, []),
    "rssm_selftest_bounded_wait": (c_int, [P, P]),
    "rssm_status_string": (c_char_p, [c_int]),
    "rssm_mamba2_ring_bytes": (c_int, [P, P]),
    "rssm_gdn_ring_bytes": (c_int, [P, P]),
    "rssm_mamba2_conventional_step": (c_int, [P] * 10 + [P]),
    "rssm_mamba2_step": (c_int, [P] * 15),
    "rssm_mamba2_flush": (c_int, [P] * 7 + [P]),
    "rssm_mamba2_spec_verify": (c_int, [P, c_int] + [P] * 14),
    "rssm_commit_cursors": (c_int, [P, P, c_int, c_int, P, P]),
    "rssm_commit_cursors_slots": (c_int, [P, P, P, c_int, c_int, c_int, P, P]),
    "rssm_reset_cursors": (c_int, [P, P, c_int, c_int, P, P]),
    "rssm_checkpoint_downcast": (c_int, [P, P, c_size_t, c_int, P]),
    "rssm_mamba2_downcast": (c_int, [P, P, P, P]),
    "rssm_gdn_conventional_step": (c_int, [P] * 8 + [P]),
    "rssm_gdn_step": (c_int, [P] * 11 + [P]),
    "rssm_gdn_flush": (c_int, [P] * 5 + [P]),
    "rssm_gdn_prime": (c_int, [P] * 5 + [P]),
    "rssm_gdn_spec_verify": (c_int, [P, c_int] + [P] * 11),
    "rssm_kda_ring_bytes": (c_int, [P, P]),
    "rssm_kda_conventional_step": (c_int, [P] * 8 + [P]),
    "rssm_kda_step": (c_int, [P] * 11 + [P]),
    "rssm_kda_flush": (c_int, [P] * 5 + [P]),
    "rssm_kda_prime": (c_int, [P] * 5 + [P]),
    "rssm_kda_spec_verify": (c_int, [P, c_int] + [P] * 11),
    "rssm_mamba2_emulated_workspace_bytes": (c_size_t, [P, P]),
    "rssm_mamba2_step_emulated": (c_int, [P] * 15 + [c_size_t, P, P]),
    "rssm_mamba2_step_emulated_noalloc": (c_int, [P] * 16),
}
EXPORTED = tuple(_SIGNATURES)

_lib = None


class RssmError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {code} ({status_string(code)})" if what else f"{code} ({status_string(code)})")


def load():
    """Load librssm.so (built in-tree); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"librssm.so is not built ({LIB_PATH}); run "
                               "`python -m recurrent_state_decode_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(code):
    return load().rssm_status_string(int(code)).decode()


def check(rc, what=""):
    if rc != RSSM_OK:
        raise RssmError(rc, what)
    return rc


def ptr(t):
    """Address of a tensor / int / None for a pointer argument."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, *tensors):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    for t in tensors:
        if hasattr(t, "is_cuda") and t.is_cuda:
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def mamba2_desc(batch, nheads, headdim, dstate, ngroups, buf_len, out_dtype=RSSM_F32, read_dtype=0,
                state_slots=None, n_slots=0):
    """state_slots: int32 [batch] state row per batch row (-1 padding), with n_slots state rows."""
    return rssm_mamba2_desc(batch, nheads, headdim, dstate, ngroups, buf_len, out_dtype, read_dtype,
                            ptr(state_slots), n_slots)


def mamba2_ring(x, z, B, C, dt):
    return rssm_mamba2_ring(ptr(x), ptr(z), ptr(B), ptr(C), ptr(dt))


def gdn_desc(batch, nheads, dk, dv, buf_len, out_dtype=RSSM_F32, state_slots=None, n_slots=0):
    return rssm_gdn_desc(batch, nheads, dk, dv, buf_len, out_dtype, ptr(state_slots), n_slots)


def gdn_ring(q, k, v, g, beta, e):
    return rssm_gdn_ring(ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(e))


def _ref(s):
    return None if s is None else ctypes.byref(s)


# ----------------------------------------------------------------------------- calls

def rssm_version():
    return load().rssm_version()


def rssm_selftest_bounded_wait(dev_status, stream=None):
    return load().rssm_selftest_bounded_wait(ptr(dev_status), _stream(stream, dev_status))


def rssm_mamba2_ring_bytes(desc):
    out = (c_size_t * 5)()
    check(load().rssm_mamba2_ring_bytes(_ref(desc), out), "rssm_mamba2_ring_bytes")
    return list(out)


def rssm_gdn_ring_bytes(desc):
    out = (c_size_t * 6)()
    check(load().rssm_gdn_ring_bytes(_ref(desc), out), "rssm_gdn_ring_bytes")
    return list(out)


def rssm_mamba2_conventional_step(desc, state, x, z, B, C, dt, A, D, y, stream=None):
    return load().rssm_mamba2_conventional_step(
        _ref(desc), ptr(state), ptr(x), ptr(z), ptr(B), ptr(C), ptr(dt), ptr(A), ptr(D), ptr(y),
        _stream(stream, state))


def rssm_mamba2_step(desc, ckpt, ckpt_read, ring, cursors, x, z, B, C, dt, A, D, y, dev_status=None, stream=None):
    return load().rssm_mamba2_step(
        _ref(desc), ptr(ckpt), ptr(ckpt_read), _ref(ring), ptr(cursors), ptr(x), ptr(z), ptr(B), ptr(C),
        ptr(dt), ptr(A), ptr(D), ptr(y), ptr(dev_status), _stream(stream, ckpt))


def rssm_mamba2_flush(desc, ckpt, ckpt_read, ring, cursors, A, dev_status=None, stream=None):
    return load().rssm_mamba2_flush(
        _ref(desc), ptr(ckpt), ptr(ckpt_read), _ref(ring), ptr(cursors), ptr(A), ptr(dev_status),
        _stream(stream, ckpt))


def rssm_mamba2_spec_verify(desc, n_new, ckpt, ckpt_read, ring, cursors, x, z, B, C, dt, A, D, y,
                            dev_status=None, stream=None):
    return load().rssm_mamba2_spec_verify(
        _ref(desc), int(n_new), ptr(ckpt), ptr(ckpt_read), _ref(ring), ptr(cursors), ptr(x), ptr(z), ptr(B),
        ptr(C), ptr(dt), ptr(A), ptr(D), ptr(y), ptr(dev_status), _stream(stream, ckpt))


def rssm_commit_cursors(cursors, kept, batch, buf_len, dev_status=None, stream=None):
    return load().rssm_commit_cursors(ptr(cursors), ptr(kept), int(batch), int(buf_len), ptr(dev_status),
                                      _stream(stream, cursors))


def rssm_commit_cursors_slots(cursors, kept, state_slots, batch, n_slots, buf_len, dev_status=None, stream=None):
    return load().rssm_commit_cursors_slots(ptr(cursors), ptr(kept), ptr(state_slots), int(batch), int(n_slots),
                                            int(buf_len), ptr(dev_status), _stream(stream, cursors))


def rssm_reset_cursors(cursors, slots, n_slots, batch, dev_status=None, stream=None):
    return load().rssm_reset_cursors(ptr(cursors), ptr(slots), int(n_slots), int(batch), ptr(dev_status),
                                     _stream(stream, cursors))


def rssm_checkpoint_downcast(src, dst, n, dtype=None, stream=None):
    if dtype is None:
        import torch
        dtype = RSSM_F16 if dst.dtype == torch.float16 else RSSM_BF16
    return load().rssm_checkpoint_downcast(ptr(src), ptr(dst), int(n), int(dtype), _stream(stream, src))


def rssm_gdn_conventional_step(desc, S, q, k, v, g, beta, o, stream=None):
    return load().rssm_gdn_conventional_step(
        _ref(desc), ptr(S), ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(o), _stream(stream, S))


def rssm_gdn_step(desc, S, ring, cursors, q, k, v, g, beta, o, dev_status=None, stream=None):
    return load().rssm_gdn_step(
        _ref(desc), ptr(S), _ref(ring), ptr(cursors), ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(o),
        ptr(dev_status), _stream(stream, S))


def rssm_gdn_flush(desc, S, ring, cursors, dev_status=None, stream=None):
    return load().rssm_gdn_flush(_ref(desc), ptr(S), _ref(ring), ptr(cursors), ptr(dev_status),
                                 _stream(stream, S))


def rssm_gdn_prime(desc, S, ring, cursors, dev_status=None, stream=None):
    return load().rssm_gdn_prime(_ref(desc), ptr(S), _ref(ring), ptr(cursors), ptr(dev_status),
                                 _stream(stream, S))


def rssm_gdn_spec_verify(desc, n_new, S, ring, cursors, q, k, v, g, beta, o, dev_status=None, stream=None):
    return load().rssm_gdn_spec_verify(
        _ref(desc), int(n_new), ptr(S), _ref(ring), ptr(cursors), ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(o),
        ptr(dev_status), _stream(stream, S))


def rssm_mamba2_downcast(desc, ckpt, ckpt_read, stream=None):
    return load().rssm_mamba2_downcast(_ref(desc), ptr(ckpt), ptr(ckpt_read), _stream(stream, ckpt))


def kda_desc(batch, nheads, dk, dv, buf_len, out_dtype=RSSM_F32, state_slots=None, n_slots=0):
    return gdn_desc(batch, nheads, dk, dv, buf_len, out_dtype, state_slots, n_slots)


def kda_ring(q, k, v, g, beta, e):
    return gdn_ring(q, k, v, g, beta, e)


def rssm_kda_ring_bytes(desc):
    out = (c_size_t * 6)()
    check(load().rssm_kda_ring_bytes(_ref(desc), out), "rssm_kda_ring_bytes")
    return list(out)


def rssm_kda_conventional_step(desc, S, q, k, v, g, beta, o, stream=None):
    return load().rssm_kda_conventional_step(
        _ref(desc), ptr(S), ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(o), _stream(stream, S))


def rssm_kda_step(desc, S, ring, cursors, q, k, v, g, beta, o, dev_status=None, stream=None):
    return load().rssm_kda_step(
        _ref(desc), ptr(S), _ref(ring), ptr(cursors), ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(o),
        ptr(dev_status), _stream(stream, S))


def rssm_kda_flush(desc, S, ring, cursors, dev_status=None, stream=None):
    return load().rssm_kda_flush(_ref(desc), ptr(S), _ref(ring), ptr(cursors), ptr(dev_status), _stream(stream, S))


def rssm_kda_spec_verify(desc, n_new, S, ring, cursors, q, k, v, g, beta, o, dev_status=None, stream=None):
    return load().rssm_kda_spec_verify(
        _ref(desc), int(n_new), ptr(S), _ref(ring), ptr(cursors), ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(o),
        ptr(dev_status), _stream(stream, S))


def rssm_kda_prime(desc, S, ring, cursors, dev_status=None, stream=None):
    return load().rssm_kda_prime(_ref(desc), ptr(S), _ref(ring), ptr(cursors), ptr(dev_status), _stream(stream, S))


def emulation(fmt, scale):
    """An emulated read precision: fmt an RSSM_EMU_* format, scale an RSSM_EMU_SCALE_* mode."""
    return rssm_emulation(int(fmt), int(scale))


def rssm_mamba2_emulated_workspace_bytes(desc):
    rc = ctypes.c_int(0)
    n = load().rssm_mamba2_emulated_workspace_bytes(_ref(desc), ctypes.byref(rc))
    check(rc.value, "rssm_mamba2_emulated_workspace_bytes")
    return int(n)


def rssm_mamba2_step_emulated(desc, emu, ckpt, ring, cursors, x, z, B, C, dt, A, D, y, err, workspace,
                              workspace_bytes, dev_status=None, stream=None):
    return load().rssm_mamba2_step_emulated(
        _ref(desc), _ref(emu), ptr(ckpt), _ref(ring), ptr(cursors), ptr(x), ptr(z), ptr(B), ptr(C), ptr(dt), ptr(A),
        ptr(D), ptr(y), ptr(err), ptr(workspace), int(workspace_bytes), ptr(dev_status), _stream(stream, ckpt))


RSSM_NOALLOC_MAX_WARPS = 262144


def rssm_mamba2_step_emulated_noalloc(desc, emu, ckpt, ring, cursors, x, z, B, C, dt, A, D, y, err, dev_status=None,
                                      stream=None):
    return load().rssm_mamba2_step_emulated_noalloc(
        _ref(desc), _ref(emu), ptr(ckpt), _ref(ring), ptr(cursors), ptr(x), ptr(z), ptr(B), ptr(C), ptr(dt), ptr(A),
        ptr(D), ptr(y), ptr(err), ptr(dev_status), _stream(stream, ckpt))
