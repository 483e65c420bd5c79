"""Seeded synthetic workloads for the ReplaySSM decode path.

This module draws inputs only: it holds none of the method's arithmetic and is
shared by the tests, the benchmark and the oracle harness. Every draw comes
from a ``torch.Generator`` on the requested device, seeded from
``(workload seed, stream name, index)`` so any step can be regenerated on its
own. Distributions (per workload):

* Mamba-2 records: x, z ~ N(0, 1) in bf16; B, C ~ N(0, 1/dstate) in bf16;
  dt = softplus(N(-2, 0.5)) in fp32. Parameters: A = -exp(U(0, 2.5)),
  D ~ N(0, 1), per head, fp32.
* Gated DeltaNet records: q, k ~ N(0, 1), L2-normalised per head in fp32,
  then bf16; v ~ N(0, 1) in bf16; g = -softplus(N(0, 1)); beta =
  sigmoid(N(0, 1)), fp32.
* Kimi Delta Attention records: q, k, v, beta as for Gated DeltaNet; g per
  key channel = -softplus(N(-1, 1.5)), fp32 (a spread of slow and fast
  channels: per-token decay from about 0.99 down to about 0.05).
* Checkpoint: zero (the tiny workload) or 0.1 * N(0, 1) in fp32.
* Initial window: per sequence a start slot and a fill count ~ U{0..L-1}
  (so flushes are staggered across the batch), the filled records drawn
  like step records.
* Speculative decode: accepted drafts a ~ U{0..T}; kept = a + 1 (the bonus
  token of the previous verify always commits).
"""
from dataclasses import dataclass, field

import torch
import torch.nn.functional as F

_STREAMS = {"params": 1, "ckpt": 2, "cursor": 3, "prefill": 4, "step": 5, "accept": 6}


def generator(device, seed, stream, index=0):
    """A generator seeded from (seed, stream, index) by a fixed integer mix."""
    s = (seed * 1_000_003 + _STREAMS[stream]) * 1_000_033 + index
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(s % (2 ** 62))
    return g


@dataclass(frozen=True)
class Mamba2Workload:
    name: str
    batch: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    buf_len: int
    steps: int
    seed: int
    zero_ckpt: bool = False
    prefill: bool = True
    drafts: int = 0          # T; 0 = autoregressive decode
    read_copy: object = False  # read copy of the checkpoint: False, True (bf16), "f16" or "f8"

    @property
    def n_new(self):
        return self.drafts + 1


@dataclass(frozen=True)
class GDNWorkload:
    name: str
    batch: int
    nheads: int
    dk: int
    dv: int
    buf_len: int
    steps: int
    seed: int
    zero_ckpt: bool = False
    prefill: bool = True
    drafts: int = 0          # T; 0 = autoregressive decode

    @property
    def n_new(self):
        return self.drafts + 1


@dataclass(frozen=True)
class KDAWorkload(GDNWorkload):
    """A Kimi Delta Attention workload: the Gated DeltaNet fields, records with
    one log decay per key channel."""


WORKLOADS = {
    "mamba2_tiny": Mamba2Workload("mamba2_tiny", 4, 8, 64, 128, 1, 16, 64, seed=1000, zero_ckpt=True, prefill=False),
    "mamba2_serving": Mamba2Workload("mamba2_serving", 256, 128, 64, 128, 8, 16, 256, seed=1001),
    "mamba2_spec": Mamba2Workload("mamba2_spec", 512, 128, 64, 128, 8, 16, 128, seed=1002, drafts=3),
    "gdn_serving": GDNWorkload("gdn_serving", 256, 32, 128, 128, 16, 256, seed=1003),
    "mamba2_bf16_read": Mamba2Workload("mamba2_bf16_read", 256, 128, 64, 128, 8, 16, 4096, seed=1004, read_copy=True),
    "mamba2_f16_read": Mamba2Workload("mamba2_f16_read", 256, 128, 64, 128, 8, 16, 4096, seed=1004, read_copy="f16"),
    "mamba2_f8_read": Mamba2Workload("mamba2_f8_read", 256, 128, 64, 128, 8, 16, 4096, seed=1004, read_copy="f8"),
    "gdn_spec": GDNWorkload("gdn_spec", 512, 32, 128, 128, 16, 128, seed=1005, drafts=3),
    "kda_serving": KDAWorkload("kda_serving", 256, 32, 128, 128, 16, 256, seed=1006),
    "kda_spec": KDAWorkload("kda_spec", 512, 32, 128, 128, 16, 128, seed=1007, drafts=3),
}


# ----------------------------------------------------------------------------- Mamba-2

def mamba2_params(w, device):
    g = generator(device, w.seed, "params")
    A = -torch.exp(torch.rand(w.nheads, generator=g, device=device) * 2.5)
    D = torch.randn(w.nheads, generator=g, device=device)
    return A.float().contiguous(), D.float().contiguous()


def mamba2_checkpoint(w, device):
    shape = (w.batch, w.nheads, w.headdim, w.dstate)
    if w.zero_ckpt:
        return torch.zeros(shape, dtype=torch.float32, device=device)
    g = generator(device, w.seed, "ckpt")
    return (0.1 * torch.randn(shape, generator=g, device=device)).float()


def initial_cursors(w, device):
    """(starts, counts) int32 [Bt]; zero unless the workload pre-fills windows."""
    if not w.prefill:
        z = torch.zeros(w.batch, dtype=torch.int32, device=device)
        return z, z.clone()
    g = generator(device, w.seed, "cursor")
    starts = torch.randint(0, w.buf_len, (w.batch,), generator=g, device=device, dtype=torch.int64)
    counts = torch.randint(0, w.buf_len, (w.batch,), generator=g, device=device, dtype=torch.int64)
    return starts.int(), counts.int()


def mamba2_records(w, stream, index, n, device):
    """n records per sequence: x,z [Bt,n,H,P] bf16; B,C [Bt,n,G,N] bf16; dt [Bt,n,H] fp32."""
    g = generator(device, w.seed, stream, index)
    Bt, H, P, N, G = w.batch, w.nheads, w.headdim, w.dstate, w.ngroups
    x = torch.randn((Bt, n, H, P), generator=g, device=device).to(torch.bfloat16)
    z = torch.randn((Bt, n, H, P), generator=g, device=device).to(torch.bfloat16)
    B = (torch.randn((Bt, n, G, N), generator=g, device=device) / N ** 0.5).to(torch.bfloat16)
    C = (torch.randn((Bt, n, G, N), generator=g, device=device) / N ** 0.5).to(torch.bfloat16)
    dt = F.softplus(torch.randn((Bt, n, H), generator=g, device=device) * 0.5 - 2.0).float()
    return {"x": x, "z": z, "B": B, "C": C, "dt": dt}


def mamba2_step_inputs(w, t, device):
    """Record of AR step t, with the draft axis squeezed: x,z [Bt,H,P] ..."""
    r = mamba2_records(w, "step", t, 1, device)
    return {k: v[:, 0].contiguous() for k, v in r.items()}


def mamba2_verify_inputs(w, t, device):
    """Records of verify step t: x,z [Bt,K,H,P], B,C [Bt,K,G,N], dt [Bt,K,H]."""
    return {k: v.contiguous() for k, v in mamba2_records(w, "step", t, w.n_new, device).items()}


def mamba2_prefill(w, device):
    """Window records drawn for the initial fill: [Bt, L-1, ...] (record j used iff j < count)."""
    return mamba2_records(w, "prefill", 0, max(w.buf_len - 1, 1), device)


def accepted_kept(w, t, device):
    """kept = a + 1 with a ~ U{0..T} per sequence, int32 [Bt]."""
    g = generator(device, w.seed, "accept", t)
    a = torch.randint(0, w.drafts + 1, (w.batch,), generator=g, device=device, dtype=torch.int64)
    return (a + 1).int()


# ----------------------------------------------------------------------------- Gated DeltaNet

def gdn_checkpoint(w, device):
    shape = (w.batch, w.nheads, w.dv, w.dk)
    if w.zero_ckpt:
        return torch.zeros(shape, dtype=torch.float32, device=device)
    g = generator(device, w.seed, "ckpt")
    return (0.1 * torch.randn(shape, generator=g, device=device)).float()


def gdn_records(w, stream, index, n, device):
    """q,k [Bt,n,H,dk] bf16 (unit norm before rounding); v [Bt,n,H,dv] bf16; g,beta [Bt,n,H] fp32."""
    gen = generator(device, w.seed, stream, index)
    Bt, H = w.batch, w.nheads
    q = torch.randn((Bt, n, H, w.dk), generator=gen, device=device)
    k = torch.randn((Bt, n, H, w.dk), generator=gen, device=device)
    q = (q / q.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn((Bt, n, H, w.dv), generator=gen, device=device).to(torch.bfloat16)
    g = (-F.softplus(torch.randn((Bt, n, H), generator=gen, device=device))).float()
    beta = torch.sigmoid(torch.randn((Bt, n, H), generator=gen, device=device)).float()
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta}


def gdn_step_inputs(w, t, device):
    r = gdn_records(w, "step", t, 1, device)
    return {k: v[:, 0].contiguous() for k, v in r.items()}


def gdn_verify_inputs(w, t, device):
    """Records of verify step t: q,k [Bt,K,H,dk], v [Bt,K,H,dv] bf16; g,beta [Bt,K,H] fp32."""
    return {k: v.contiguous() for k, v in gdn_records(w, "step", t, w.n_new, device).items()}


def gdn_prefill(w, device):
    return gdn_records(w, "prefill", 0, max(w.buf_len - 1, 1), device)


# ----------------------------------------------------------------------------- Kimi Delta Attention

def kda_records(w, stream, index, n, device):
    """q,k [Bt,n,H,dk] bf16 (unit norm before rounding); v [Bt,n,H,dv] bf16;
    g [Bt,n,H,dk] fp32 (per key channel); beta [Bt,n,H] fp32."""
    gen = generator(device, w.seed, stream, index)
    Bt, H = w.batch, w.nheads
    q = torch.randn((Bt, n, H, w.dk), generator=gen, device=device)
    k = torch.randn((Bt, n, H, w.dk), generator=gen, device=device)
    q = (q / q.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn((Bt, n, H, w.dv), generator=gen, device=device).to(torch.bfloat16)
    g = (-F.softplus(torch.randn((Bt, n, H, w.dk), generator=gen, device=device) * 1.5 - 1.0)).float()
    beta = torch.sigmoid(torch.randn((Bt, n, H), generator=gen, device=device)).float()
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta}


def kda_step_inputs(w, t, device):
    r = kda_records(w, "step", t, 1, device)
    return {k: v[:, 0].contiguous() for k, v in r.items()}


def kda_verify_inputs(w, t, device):
    """Records of verify step t: q,k [Bt,K,H,dk], v [Bt,K,H,dv] bf16; g [Bt,K,H,dk], beta [Bt,K,H] fp32."""
    return {k: v.contiguous() for k, v in kda_records(w, "step", t, w.n_new, device).items()}


def kda_prefill(w, device):
    return kda_records(w, "prefill", 0, max(w.buf_len - 1, 1), device)


# ----------------------------------------------------------------------------- ring placement

def place_window(ring_field, records, starts, counts, L):
    """Copy record j of sequence b into ring slot (start_b + j) mod L for j < count_b.

    ring_field [Bt, X, L, ...] (X = heads or groups); records [Bt, n, X, ...].
    Plain data placement used to set up an initial window.
    """
    n = records.shape[1]
    dev = ring_field.device
    starts = starts.long().to(dev)
    counts = counts.long().to(dev)
    for j in range(n):
        bs = torch.nonzero(counts > j).flatten()
        if bs.numel() == 0:
            break
        ring_field[bs, :, (starts[bs] + j) % L] = records[bs, j].to(ring_field.dtype)
    return ring_field


def to_f64(t):
    """Exact widening of a bf16/fp32 tensor to a float64 numpy array."""
    return t.detach().float().cpu().double().numpy()
