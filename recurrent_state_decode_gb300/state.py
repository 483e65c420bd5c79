"""Device buffers of a decode session, allocated with torch, and thin methods
that pass them to the C-ABI calls.

Plumbing only: torch owns the memory and the stream, every step runs in
librssm's kernels. Layouts follow ``include/rssm.h``.
"""
import torch

from . import binding as bd


def _check_slots(slots, like):
    """A slot table is a contiguous int32 tensor on the state's device."""
    if slots.dtype != torch.int32 or slots.device != like.device or not slots.is_contiguous():
        raise ValueError(f"state slots must be a contiguous int32 tensor on {like.device}, "
                         f"got {slots.dtype} on {slots.device}")


def _check_tensor(name, t, dtype, shape, device):
    """A tensor argument is a contiguous tensor of the given dtype and shape on
    the state's device: the C ABI reads it by its base pointer alone."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor, got {type(t).__name__}")
    shape = tuple(int(v) for v in shape)
    if t.dtype != dtype or t.device != device or tuple(t.shape) != shape or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {shape} on {device}, got {t.dtype} "
                         f"{tuple(t.shape)} on {t.device}{'' if t.is_contiguous() else ' (not contiguous)'}")


def _check_records(rec, spec, rows, device, n_new=None):
    """Record fields against their (dtype, per-row shape); n_new adds the draft axis."""
    lead = (rows,) if n_new is None else (rows, n_new)
    for name, (dtype, tail) in spec.items():
        if name not in rec:
            raise ValueError(f"record field {name} is missing")
        _check_tensor(name, rec[name], dtype, lead + tail, device)


def _draft_count(rec, field):
    t = rec.get(field)
    if not isinstance(t, torch.Tensor) or t.dim() < 2 or t.shape[1] < 1:
        raise ValueError(f"{field} of a verify must have a draft axis [rows, K, ...] with K >= 1")
    return int(t.shape[1])


class Mamba2State:
    """Checkpoint (+ optional read copy: read_copy True or "bf16" for bf16,
    "f16" for fp16, "f8" for e4m3 with one fp32 scale per state row), ring
    buffer, cursors and a device status word for one Mamba-2 layer of
    `batch` sequences.

    The decode calls take an optional ``slots`` (int32 [rows] on the device):
    batch row r then uses state row slots[r] of this object's ``batch`` rows
    (-1: a padding row, skipped), and records / outputs have ``rows`` rows."""

    def __init__(self, batch, nheads, headdim, dstate, ngroups, buf_len, device="cuda",
                 read_copy=False, out_dtype=bd.RSSM_F32):
        self.batch, self.nheads, self.headdim, self.dstate = batch, nheads, headdim, dstate
        self.ngroups, self.buf_len, self.out_dtype = ngroups, buf_len, out_dtype
        f16, f8 = read_copy == "f16", read_copy == "f8"
        self.desc = bd.mamba2_desc(batch, nheads, headdim, dstate, ngroups, buf_len, out_dtype,
                                   bd.RSSM_FP8_E4M3 if f8 else (bd.RSSM_F16 if f16 else bd.RSSM_BF16))
        dev = torch.device(device)
        self.ckpt = torch.zeros((batch, nheads, headdim, dstate), dtype=torch.float32, device=dev)
        if f8:  # e4m3 bytes, then one fp32 scale per state row
            n, rows = batch * nheads * headdim * dstate, batch * nheads * headdim
            self.ckpt_read = torch.zeros(n + 4 * rows, dtype=torch.uint8, device=dev)
            self.read_q = self.ckpt_read[:n].view(batch, nheads, headdim, dstate)
            self.read_scale = self.ckpt_read[n:].view(torch.float32).view(batch, nheads, headdim)
        else:
            self.ckpt_read = (torch.zeros((batch, nheads, headdim, dstate),
                                          dtype=torch.float16 if f16 else torch.bfloat16, device=dev)
                              if read_copy else None)
        self.rx = torch.zeros((batch, nheads, buf_len, headdim), dtype=torch.bfloat16, device=dev)
        self.rz = torch.zeros_like(self.rx)
        self.rB = torch.zeros((batch, ngroups, buf_len, dstate), dtype=torch.bfloat16, device=dev)
        self.rC = torch.zeros_like(self.rB)
        self.rdt = torch.zeros((batch, nheads, (buf_len + 3) // 4 * 4), dtype=torch.float32, device=dev)
        self.ring = bd.mamba2_ring(self.rx, self.rz, self.rB, self.rC, self.rdt)
        self.cursors = torch.zeros((batch, 4), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    @property
    def y_dtype(self):
        return torch.bfloat16 if self.out_dtype == bd.RSSM_BF16 else torch.float32

    def new_output(self, n_new=0, rows=None):
        rows = self.batch if rows is None else rows
        shape = (rows, self.nheads, self.headdim) if n_new == 0 else (rows, n_new, self.nheads, self.headdim)
        return torch.empty(shape, dtype=self.y_dtype, device=self.ckpt.device)

    def slot_desc(self, slots):
        """The descriptor of a call whose batch rows use state rows ``slots``."""
        _check_slots(slots, self.ckpt)
        d = self.desc
        return bd.mamba2_desc(slots.numel(), d.nheads, d.headdim, d.dstate, d.ngroups, d.buf_len, d.out_dtype,
                              d.read_dtype, state_slots=slots, n_slots=self.batch)

    def downcast(self, stream=None):
        bd.check(bd.rssm_mamba2_downcast(self.desc, self.ckpt, self.ckpt_read, stream), "rssm_mamba2_downcast")

    def _record_spec(self):
        H, P, N, G = self.nheads, self.headdim, self.dstate, self.ngroups
        bf, f32 = torch.bfloat16, torch.float32
        return {"x": (bf, (H, P)), "z": (bf, (H, P)), "B": (bf, (G, N)), "C": (bf, (G, N)), "dt": (f32, (H,))}

    def _check_params(self, A, D=None):
        dev = self.ckpt.device
        _check_tensor("A", A, torch.float32, (self.nheads,), dev)
        if D is not None:
            _check_tensor("D", D, torch.float32, (self.nheads,), dev)

    def step(self, rec, A, D, y, stream=None, slots=None):
        desc = self.desc if slots is None else self.slot_desc(slots)
        dev = self.ckpt.device
        _check_records(rec, self._record_spec(), desc.batch, dev)
        self._check_params(A, D)
        _check_tensor("y", y, self.y_dtype, (desc.batch, self.nheads, self.headdim), dev)
        bd.check(bd.rssm_mamba2_step(desc, self.ckpt, self.ckpt_read, self.ring, self.cursors,
                                     rec["x"], rec["z"], rec["B"], rec["C"], rec["dt"], A, D, y,
                                     self.status, stream), "rssm_mamba2_step")

    def step_emulated(self, rec, A, D, y, emu, err, workspace, stream=None):
        """rssm_mamba2_step with an emulated read precision: emu from
        ``binding.emulation``; err float64 [2] and workspace (uint8, at least
        ``binding.rssm_mamba2_emulated_workspace_bytes(self.desc)`` bytes) on
        the device."""
        dev = self.ckpt.device
        _check_records(rec, self._record_spec(), self.batch, dev)
        self._check_params(A, D)
        _check_tensor("y", y, self.y_dtype, (self.batch, self.nheads, self.headdim), dev)
        _check_tensor("err", err, torch.float64, (2,), dev)
        if not isinstance(workspace, torch.Tensor) or workspace.device != dev or not workspace.is_contiguous():
            raise ValueError(f"workspace must be a contiguous tensor on {dev}")
        nbytes = workspace.numel() * workspace.element_size()
        bd.check(bd.rssm_mamba2_step_emulated(self.desc, emu, self.ckpt, self.ring, self.cursors, rec["x"], rec["z"],
                                              rec["B"], rec["C"], rec["dt"], A, D, y, err, workspace, nbytes,
                                              self.status, stream), "rssm_mamba2_step_emulated")

    def flush(self, A, stream=None):
        self._check_params(A)
        bd.check(bd.rssm_mamba2_flush(self.desc, self.ckpt, self.ckpt_read, self.ring, self.cursors, A,
                                      self.status, stream), "rssm_mamba2_flush")

    def verify(self, rec, A, D, y, stream=None, slots=None):
        n_new = _draft_count(rec, "x")
        desc = self.desc if slots is None else self.slot_desc(slots)
        dev = self.ckpt.device
        _check_records(rec, self._record_spec(), desc.batch, dev, n_new)
        self._check_params(A, D)
        _check_tensor("y", y, self.y_dtype, (desc.batch, n_new, self.nheads, self.headdim), dev)
        bd.check(bd.rssm_mamba2_spec_verify(desc, n_new, self.ckpt, self.ckpt_read, self.ring, self.cursors,
                                            rec["x"], rec["z"], rec["B"], rec["C"], rec["dt"], A, D, y,
                                            self.status, stream), "rssm_mamba2_spec_verify")

    def commit(self, kept, stream=None, slots=None):
        _commit(self, kept, stream, slots)

    def reset(self, slots, stream=None):
        _check_slots(slots, self.cursors)
        bd.check(bd.rssm_reset_cursors(self.cursors, slots, slots.numel(), self.batch, self.status, stream),
                 "rssm_reset_cursors")


def _commit(st, kept, stream, slots):
    if slots is not None:
        _check_slots(slots, st.cursors)
    _check_tensor("kept", kept, torch.int32, (st.batch if slots is None else slots.numel(),), st.cursors.device)
    if slots is None:
        bd.check(bd.rssm_commit_cursors(st.cursors, kept, st.batch, st.buf_len, st.status, stream),
                 "rssm_commit_cursors")
    else:
        bd.check(bd.rssm_commit_cursors_slots(st.cursors, kept, slots, slots.numel(), st.batch, st.buf_len,
                                              st.status, stream), "rssm_commit_cursors_slots")


class GDNState:
    """Checkpoint S, ring buffer, cursors and status word for one Gated DeltaNet
    layer; ``slots`` on the decode calls as in Mamba2State."""

    def __init__(self, batch, nheads, dk, dv, buf_len, device="cuda", out_dtype=bd.RSSM_F32):
        self.batch, self.nheads, self.dk, self.dv, self.buf_len = batch, nheads, dk, dv, buf_len
        self.out_dtype = out_dtype
        self.desc = bd.gdn_desc(batch, nheads, dk, dv, buf_len, out_dtype)
        dev = torch.device(device)
        self.S = torch.zeros((batch, nheads, dv, dk), dtype=torch.float32, device=dev)
        self.rq = torch.zeros((batch, nheads, buf_len, dk), dtype=torch.bfloat16, device=dev)
        self.rk = torch.zeros_like(self.rq)
        self.rv = torch.zeros((batch, nheads, buf_len, dv), dtype=torch.bfloat16, device=dev)
        self.rg = torch.zeros((batch, nheads, (buf_len + 3) // 4 * 4), dtype=torch.float32, device=dev)
        self.rbeta = torch.zeros_like(self.rg)
        self.re = torch.zeros((batch, nheads, buf_len, dv), dtype=torch.float32, device=dev)
        self.ring = bd.gdn_ring(self.rq, self.rk, self.rv, self.rg, self.rbeta, self.re)
        self.cursors = torch.zeros((batch, 4), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    @property
    def o_dtype(self):
        return torch.bfloat16 if self.out_dtype == bd.RSSM_BF16 else torch.float32

    def new_output(self, rows=None):
        rows = self.batch if rows is None else rows
        return torch.empty((rows, self.nheads, self.dv), dtype=self.o_dtype, device=self.S.device)

    def slot_desc(self, slots):
        _check_slots(slots, self.S)
        d = self.desc
        return bd.gdn_desc(slots.numel(), d.nheads, d.dk, d.dv, d.buf_len, d.out_dtype, state_slots=slots,
                           n_slots=self.batch)

    def _record_spec(self):
        H, bf, f32 = self.nheads, torch.bfloat16, torch.float32
        return {"q": (bf, (H, self.dk)), "k": (bf, (H, self.dk)), "v": (bf, (H, self.dv)), "g": (f32, (H,)),
                "beta": (f32, (H,))}

    def _check_call(self, rec, o, desc, n_new=None):
        dev = self.S.device
        _check_records(rec, self._record_spec(), desc.batch, dev, n_new)
        lead = (desc.batch,) if n_new is None else (desc.batch, n_new)
        _check_tensor("o", o, self.o_dtype, lead + (self.nheads, self.dv), dev)

    def step(self, rec, o, stream=None, slots=None):
        desc = self.desc if slots is None else self.slot_desc(slots)
        self._check_call(rec, o, desc)
        bd.check(bd.rssm_gdn_step(desc, self.S, self.ring, self.cursors, rec["q"], rec["k"], rec["v"],
                                  rec["g"], rec["beta"], o, self.status, stream), "rssm_gdn_step")

    def flush(self, stream=None):
        bd.check(bd.rssm_gdn_flush(self.desc, self.S, self.ring, self.cursors, self.status, stream),
                 "rssm_gdn_flush")

    def new_verify_output(self, n_new, rows=None):
        rows = self.batch if rows is None else rows
        return torch.empty((rows, n_new, self.nheads, self.dv), dtype=self.o_dtype, device=self.S.device)

    def verify(self, rec, o, stream=None, slots=None):
        """rec: q,k [Bt,K,H,dk], v [Bt,K,H,dv] bf16; g,beta [Bt,K,H] fp32; o [Bt,K,H,dv]."""
        desc = self.desc if slots is None else self.slot_desc(slots)
        n_new = _draft_count(rec, "q")
        self._check_call(rec, o, desc, n_new)
        bd.check(bd.rssm_gdn_spec_verify(desc, n_new, self.S, self.ring, self.cursors, rec["q"],
                                         rec["k"], rec["v"], rec["g"], rec["beta"], o, self.status, stream),
                 "rssm_gdn_spec_verify")

    def commit(self, kept, stream=None, slots=None):
        _commit(self, kept, stream, slots)

    def prime(self, stream=None):
        """Fill the ring's corrections e for records placed into the window directly."""
        bd.check(bd.rssm_gdn_prime(self.desc, self.S, self.ring, self.cursors, self.status, stream),
                 "rssm_gdn_prime")


class KDAState(GDNState):
    """Checkpoint S, ring buffer (g with one log decay per key channel), cursors
    and status word for one Kimi Delta Attention layer."""

    def __init__(self, batch, nheads, dk, dv, buf_len, device="cuda", out_dtype=bd.RSSM_F32):
        super().__init__(batch, nheads, dk, dv, buf_len, device, out_dtype)
        self.rg = torch.zeros((batch, nheads, buf_len, dk), dtype=torch.float32, device=self.S.device)
        self.ring = bd.kda_ring(self.rq, self.rk, self.rv, self.rg, self.rbeta, self.re)

    def _record_spec(self):
        spec = super()._record_spec()
        spec["g"] = (torch.float32, (self.nheads, self.dk))
        return spec

    def step(self, rec, o, stream=None, slots=None):
        desc = self.desc if slots is None else self.slot_desc(slots)
        self._check_call(rec, o, desc)
        bd.check(bd.rssm_kda_step(desc, self.S, self.ring, self.cursors, rec["q"], rec["k"], rec["v"],
                                  rec["g"], rec["beta"], o, self.status, stream), "rssm_kda_step")

    def flush(self, stream=None):
        bd.check(bd.rssm_kda_flush(self.desc, self.S, self.ring, self.cursors, self.status, stream),
                 "rssm_kda_flush")

    def prime(self, stream=None):
        """Fill the ring's corrections e for records placed into the window directly."""
        bd.check(bd.rssm_kda_prime(self.desc, self.S, self.ring, self.cursors, self.status, stream),
                 "rssm_kda_prime")

    def verify(self, rec, o, stream=None, slots=None):
        """rec: q,k [Bt,K,H,dk], v [Bt,K,H,dv] bf16; g [Bt,K,H,dk], beta [Bt,K,H] fp32; o [Bt,K,H,dv]."""
        desc = self.desc if slots is None else self.slot_desc(slots)
        n_new = _draft_count(rec, "q")
        self._check_call(rec, o, desc, n_new)
        bd.check(bd.rssm_kda_spec_verify(desc, n_new, self.S, self.ring, self.cursors, rec["q"],
                                         rec["k"], rec["v"], rec["g"], rec["beta"], o, self.status, stream),
                 "rssm_kda_spec_verify")


def mamba2_from_workload(w, device="cuda", out_dtype=bd.RSSM_F32, read_copy=None):
    """A Mamba2State at the start of workload ``w`` (see ``inputs``): checkpoint,
    pre-filled windows and cursors; the read copy is downcast if present.
    Returns (state, A, D, prefill records, starts, counts)."""
    from . import inputs as I
    read_copy = w.read_copy if read_copy is None else read_copy
    st = Mamba2State(w.batch, w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len, device,
                     read_copy=read_copy, out_dtype=out_dtype)
    A, D = I.mamba2_params(w, device)
    st.ckpt.copy_(I.mamba2_checkpoint(w, device))
    starts, counts = I.initial_cursors(w, device)
    pre = I.mamba2_prefill(w, device)
    for field, ring in (("x", st.rx), ("z", st.rz), ("B", st.rB), ("C", st.rC), ("dt", st.rdt)):
        I.place_window(ring, pre[field], starts, counts, w.buf_len)
    st.cursors[:, 0] = starts
    st.cursors[:, 1] = counts
    if read_copy:
        st.downcast()
    return st, A, D, pre, starts, counts


def gdn_from_workload(w, device="cuda", out_dtype=bd.RSSM_F32):
    """A GDNState at the start of workload ``w``. Returns (state, prefill, starts, counts)."""
    from . import inputs as I
    st = GDNState(w.batch, w.nheads, w.dk, w.dv, w.buf_len, device, out_dtype=out_dtype)
    st.S.copy_(I.gdn_checkpoint(w, device))
    starts, counts = I.initial_cursors(w, device)
    pre = I.gdn_prefill(w, device)
    for field, ring in (("q", st.rq), ("k", st.rk), ("v", st.rv), ("g", st.rg), ("beta", st.rbeta)):
        I.place_window(ring, pre[field], starts, counts, w.buf_len)
    st.cursors[:, 0] = starts
    st.cursors[:, 1] = counts
    st.prime()
    return st, pre, starts, counts


def kda_from_workload(w, device="cuda", out_dtype=bd.RSSM_F32):
    """A KDAState at the start of workload ``w``. Returns (state, prefill, starts, counts)."""
    from . import inputs as I
    st = KDAState(w.batch, w.nheads, w.dk, w.dv, w.buf_len, device, out_dtype=out_dtype)
    st.S.copy_(I.gdn_checkpoint(w, device))
    starts, counts = I.initial_cursors(w, device)
    pre = I.kda_prefill(w, device)
    for field, ring in (("q", st.rq), ("k", st.rk), ("v", st.rv), ("g", st.rg), ("beta", st.rbeta)):
        I.place_window(ring, pre[field], starts, counts, w.buf_len)
    st.cursors[:, 0] = starts
    st.cursors[:, 1] = counts
    st.prime()
    return st, pre, starts, counts
