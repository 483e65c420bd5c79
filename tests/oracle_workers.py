"""Oracle decode sessions in worker processes, one chunk of sequences each,
for parity checks over whole batches at the benchmark's sizes.

Sequences are independent, so a batch's oracle session is the sessions of
its chunks. Each worker (a spawned process: started with nothing of CUDA in
it, it imports only numpy and ``oracle``) owns one chunk's session, receives
every step's records and the GPU's outputs for its sequences through a pipe,
advances its session and reduces the comparison to a few numbers per step; at
the end it compares the GPU's final checkpoints with the states at each
sequence's last flush or fold. The parent streams steps while the GPU runs,
so host memory holds one step at a time.
"""
import multiprocessing as mp
import os

import numpy as np


def half_ulp_bf16(v):
    """Half a bf16 unit in the last place of |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def out_stats(y_gpu, y_ref):
    """What a step's output comparison needs from one chunk: sums of squares of
    the difference and of the reference, their element count, and the largest
    excess of |difference| over half a bf16 ulp of the reference."""
    y_gpu = np.asarray(y_gpu, np.float64)
    d = y_gpu - y_ref
    return (float(np.sum(d * d)), float(np.sum(y_ref * y_ref)), int(y_ref.size),
            float(np.max(np.abs(d) - half_ulp_bf16(y_ref))), bool(np.isfinite(y_gpu).all()))


class _Feed:
    def __init__(self):
        self.value = None

    def __iter__(self):
        while True:
            yield self.value


def _session(kind, init, fv, fk):
    from oracle import sessions
    L = init["L"]
    pre, starts, counts = init["prefill"], init["starts"], init["counts"]
    if kind == "mamba2_ar":
        return sessions.mamba2_ar_session(init["h0"], pre, starts, counts, fv, init["A"], init["D"], L), "y"
    if kind == "mamba2_spec":
        return sessions.mamba2_spec_session(init["h0"], pre, starts, counts, fv, fk, init["A"], init["D"], L), "y"
    if kind == "gdn_ar":
        return sessions.gdn_ar_session(init["h0"], pre, starts, counts, fv, L), "o"
    if kind == "gdn_spec":
        return sessions.gdn_spec_session(init["h0"], pre, starts, counts, fv, fk, L), "o"
    if kind == "kda_ar":
        return sessions.kda_ar_session(init["h0"], pre, starts, counts, fv, L), "o"
    if kind == "kda_spec":
        return sessions.kda_spec_session(init["h0"], pre, starts, counts, fv, fk, L), "o"
    raise ValueError(kind)


def _worker(conn, kind, init):
    fv, fk = _Feed(), _Feed()
    sess, out_key = _session(kind, init, fv, fk)
    spec = kind.endswith("_spec")
    last = {}          # sequence -> state at its latest flush (AR) or fold (spec)
    stats = []
    while True:
        msg = conn.recv()
        if msg[0] == "final":
            ckpt = msg[1]
            errs = {int(i): rel_l2(ckpt[i], s) for i, s in last.items()}
            conn.send((stats, errs))
            return
        _, rec, kept, out = msg
        fv.value, fk.value = rec, kept
        exp = next(sess)
        stats.append(out_stats(out, exp[out_key]) if out is not None else None)
        hit = exp["folded"] if spec else exp["flushed"]
        for i in np.nonzero(hit)[0]:
            last[int(i)] = exp["committed_state" if spec else "state"][i].copy()


class OraclePool:
    """One spawned worker per chunk of a batch's sequences.

    chunks: list of index arrays; init_of(chunk) -> the session's initial data
    for those sequences (h0, prefill, starts, counts, L and the layer's
    parameters, as numpy)."""

    def __init__(self, kind, chunks, init_of):
        ctx = mp.get_context("spawn")
        self.chunks = chunks
        self.conns, self.procs = [], []
        for c in chunks:
            a, b = ctx.Pipe()
            p = ctx.Process(target=_worker, args=(b, kind, init_of(c)), daemon=True)
            p.start()
            b.close()
            self.conns.append(a)
            self.procs.append(p)

    def step(self, rec_of, kept_of=None, out_of=None):
        """Send one step: rec_of(chunk) -> records, kept_of(chunk) -> kept
        (spec), out_of(chunk) -> the GPU's outputs or None (not compared)."""
        for c, conn in zip(self.chunks, self.conns):
            conn.send(("step", rec_of(c), None if kept_of is None else kept_of(c),
                       None if out_of is None else out_of(c)))

    def finish(self, ckpt_of):
        """Send each chunk's final GPU checkpoint; returns per-step output errors
        over the whole batch and the checkpoint errors of every sequence that
        flushed or folded: (rel_l2 [steps], bf16_excess [steps], finite [steps],
        {sequence: rel_l2})."""
        for c, conn in zip(self.chunks, self.conns):
            conn.send(("final", ckpt_of(c)))
        results = [conn.recv() for conn in self.conns]
        for p in self.procs:
            p.join(timeout=60)
        steps = len(results[0][0])
        rel, excess, finite = [], [], []
        for t in range(steps):
            parts = [r[0][t] for r in results]
            if parts[0] is None:
                rel.append(None), excess.append(None), finite.append(None)
                continue
            sd, sr, n = sum(p[0] for p in parts), sum(p[1] for p in parts), sum(p[2] for p in parts)
            rms = np.sqrt(sr / n)
            rel.append(float(np.sqrt(sd / sr)) if sr > 0 else float(np.sqrt(sd)))
            excess.append(max(p[3] for p in parts) / rms if rms > 0 else 0.0)
            finite.append(all(p[4] for p in parts))
        ck = {}
        for c, r in zip(self.chunks, results):
            for i, e in r[1].items():
                ck[int(c[i])] = e
        return rel, excess, finite, ck

    def close(self):
        for p in self.procs:
            if p.is_alive():
                p.kill()


def chunks_of(n, parts=None):
    """n sequence indices split into about one chunk per host core."""
    parts = min(n, parts or os.cpu_count() or 1)
    return [c for c in np.array_split(np.arange(n), parts) if len(c)]
