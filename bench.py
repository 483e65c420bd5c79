#!/usr/bin/env python3
"""Benchmark of the ReplaySSM decode path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mamba2_serving|mamba2_spec|gdn_serving|gdn_spec|kda_serving|kda_spec|mamba2_bf16_read|mamba2_f16_read|mamba2_f8_read|mamba2_tiny]
    python bench.py --mode profile --steps 3 --warmup 1      # a few calls, no timing (for ncu)

A step is one decode step of one layer over the whole batch: one
``rssm_mamba2_step`` call (the append, the output-only read of the checkpoint
and window, the flush fused into every sequence's L-th step, the cursor
advance). Inputs are resident in HBM before the timed region; the 1 GiB
checkpoint streamed each step is larger than L2, so no flush is needed. The
same steps also run through the in-house conventional kernel (read + write of
the full state every step) for the speedup.

Prints ONE JSON line (rank 0). Under torchrun every rank runs its own replica
(sequences shard with no exchange: weak scaling), timing is the max over
ranks, and value/tokens are whole-job figures.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Mamba2 ReplaySSM decode µs/step/layer & HBM GB/s at B=256,L=16 vs conventional"
UNIT = "us/step/layer"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300's HBM3e as quoted (~8 TB/s); the graded fraction uses the measured copy peak


# ----------------------------------------------------------------------------- plumbing

def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mamba2_serving")
    ap.add_argument("--mode", choices=["bench", "profile"], default="bench")
    ap.add_argument("--out-dtype", choices=["bf16", "f32"], default="bf16")
    ap.add_argument("--cpu-seconds", type=float, default=2.0,
                    help="wall-clock seconds of oracle decoding per configuration for cpu_baseline (all host cores)")
    ap.add_argument("--detail", default=None, help="also write the full result, every workload's figures, here")
    ap.add_argument("--bytes-out", default=None,
                    help="profile mode: write the algorithmic bytes of every call it makes (JSON) here")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")  # host-side coordination only: no data-path collective
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        load = [v for v in sm if smax and v >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_file, kernel_sources):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", profile_file)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != source_hash(kernel_sources):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


KERNEL_SOURCES = ["recurrent_state_decode_gb300/csrc/mamba2_step_fast.cu",
                  "recurrent_state_decode_gb300/csrc/fast_rows.cuh",
                  "recurrent_state_decode_gb300/csrc/common.cuh"]


# ----------------------------------------------------------------------------- oracle (CPU baseline / reference arm)

# The configurations the metric's family is quoted on, in order: the tiny
# parity case, the serving layer (the metric's), the speculative layer, the
# Gated DeltaNet layer and the serving layer with a bf16 read copy.
CPU_CONFIGS = ["mamba2_tiny", "mamba2_serving", "mamba2_spec", "gdn_serving", "mamba2_bf16_read"]


def _oracle_worker(conn, kind, init, recs, kepts):
    """One host core's share of an oracle decode: the oracle's session over a
    chunk of sequences, advanced n steps per request (its records cycled);
    replies with the seconds those steps took. Runs in a spawned process
    holding numpy and the oracle only."""
    import time as _time

    from oracle import sessions

    def cycle(xs):
        i = 0
        while True:
            yield xs[i % len(xs)]
            i += 1

    L, pre, starts, counts = init["L"], init["prefill"], init["starts"], init["counts"]
    if kind == "mamba2_ar":
        sess = sessions.mamba2_ar_session(init["h0"], pre, starts, counts, cycle(recs), init["A"], init["D"], L)
    elif kind == "mamba2_spec":
        sess = sessions.mamba2_spec_session(init["h0"], pre, starts, counts, cycle(recs), cycle(kepts), init["A"],
                                            init["D"], L)
    else:
        sess = sessions.gdn_ar_session(init["h0"], pre, starts, counts, cycle(recs), L)
    next(sess)  # the window's replay from the checkpoint and a first step stay outside any timing
    conn.send("ready")
    while True:
        n = conn.recv()
        if n is None:
            return
        t0 = _time.perf_counter()
        for _ in range(n):
            next(sess)
        conn.send(_time.perf_counter() - t0)


class CpuOracle:
    """The oracle's fp64 decode of the first `nseq` sequences of workload `w`,
    split over `procs` spawned worker processes (one per host core); a step
    is one decode step (one verify + commit for a speculative workload) of
    every sampled sequence. Inputs are drawn beforehand (on the GPU when there
    is one) and cycled."""

    POOL = 8  # distinct steps of records, cycled

    def __init__(self, w, nseq, procs):
        import multiprocessing as mp

        import numpy as np
        import torch

        from recurrent_state_decode_gb300 import inputs as I
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        self.w, self.nseq = w, min(nseq, w.batch)
        s = slice(0, self.nseq)

        def np_(t):
            return t[s].detach().float().cpu().numpy()

        gdn = hasattr(w, "dk")
        spec = w.drafts > 0
        self.kind = "gdn_ar" if gdn else ("mamba2_spec" if spec else "mamba2_ar")
        starts, counts = (t[s].cpu().numpy() for t in I.initial_cursors(w, dev))
        if gdn:
            h0, pre = np_(I.gdn_checkpoint(w, dev)), {k: np_(v) for k, v in I.gdn_prefill(w, dev).items()}
            params = {}
            recs = [{k: np_(v) for k, v in I.gdn_step_inputs(w, t, dev).items()} for t in range(self.POOL)]
        else:
            h0 = np_(I.mamba2_checkpoint(w, dev))
            pre = {k: np_(v) for k, v in I.mamba2_prefill(w, dev).items()} if w.prefill else None
            A, D = I.mamba2_params(w, dev)
            params = {"A": A.cpu().numpy(), "D": D.cpu().numpy()}
            step = I.mamba2_verify_inputs if spec else I.mamba2_step_inputs
            recs = [{k: np_(v) for k, v in step(w, t, dev).items()} for t in range(self.POOL)]
        kepts = [I.accepted_kept(w, t, dev)[s].cpu().numpy() for t in range(self.POOL)] if spec else None
        parts = [c for c in np.array_split(np.arange(self.nseq), max(1, min(procs, self.nseq))) if len(c)]
        self.procs = len(parts)
        ctx = mp.get_context("spawn")
        self.conns, self.workers = [], []
        for c in parts:
            cs = slice(int(c[0]), int(c[-1]) + 1)
            init = {"h0": h0[cs], "prefill": None if pre is None else {k: v[cs] for k, v in pre.items()},
                    "starts": starts[cs], "counts": counts[cs], "L": w.buf_len, **params}
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, daemon=True,
                            args=(b, self.kind, init, [{k: v[cs] for k, v in r.items()} for r in recs],
                                  None if kepts is None else [k[cs] for k in kepts]))
            p.start()
            b.close()
            self.conns.append(a)
            self.workers.append(p)
        for a in self.conns:
            assert a.recv() == "ready"

    def run(self, n):
        """Wall-clock seconds for n steps of the whole sample on all workers."""
        t0 = time.perf_counter()
        for a in self.conns:
            a.send(n)
        for a in self.conns:
            a.recv()
        return time.perf_counter() - t0

    def us_per_full_step(self, seconds, n):
        """µs per decode step of the full batch on these cores."""
        return seconds / n * (self.w.batch / self.nseq) * 1e6

    def describe(self, n, seconds):
        what = "verify + commit" if self.kind == "mamba2_spec" else "decode"
        return (f"oracle conventional fp64 {what} (numpy) of {self.nseq} of {self.w.batch} sequences on "
                f"{self.procs} worker processes, {n} steps in {seconds:.2f} s, scaled to the full batch")

    def close(self):
        for a in self.conns:
            try:
                a.send(None)
            except Exception:
                pass
        for p in self.workers:
            p.join(timeout=10)
            if p.is_alive():
                p.kill()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample_size(w, cores):
    """Sequences in a bounded sample: the whole batch when small, else two per core, at least 32."""
    return min(w.batch, max(32, 2 * cores))


def oracle_baseline(name, budget_s, cores):
    """The oracle timed on workload `name`: µs per full-batch step and its sample."""
    from recurrent_state_decode_gb300 import inputs as I
    w = I.WORKLOADS[name]
    r = CpuOracle(w, oracle_sample_size(w, cores), cores)
    try:
        n, sec = 1, r.run(1)
        while sec < budget_s and n < 4096:   # grow the step count until the budget is reached
            n = max(n + 1, int(n * min(8.0, budget_s / max(sec, 1e-3))))
            sec = r.run(n)
        return r.us_per_full_step(sec, n), r.describe(n, sec), r.procs
    finally:
        r.close()


def cpu_baselines(main_name, budget_s):
    """The oracle on every configuration of CPU_CONFIGS (plus the bench's own
    workload), each for about budget_s seconds on all host cores; the bench
    workload's entry is the top-level cpu_baseline, the others ride in
    per_config."""
    cores = host_cores()
    per, top = {}, None
    names = CPU_CONFIGS + ([main_name] if main_name not in CPU_CONFIGS else [])
    for name in names:
        v, sample, used = oracle_baseline(name, budget_s, cores)
        per[name] = {"value": round(v, 1), "cores": used}
        if name == main_name:
            top = {"value": v, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample}
    top["per_config"] = per
    top["per_config_unit"] = "us per full-batch step (verify + commit for mamba2_spec), fp64 oracle"
    return top


def run_reference(args, dist):
    """The reference arm: the oracle as it stands, on the host cores. Each
    bench step is one oracle decode step of a bounded sample of sequences,
    split over all host cores, scaled to the full batch."""
    if dist.rank != 0:
        return None
    from recurrent_state_decode_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    cores = host_cores()
    r = CpuOracle(w, oracle_sample_size(w, cores), cores)
    try:
        if args.warmup:
            r.run(args.warmup)
        dt = r.run(args.steps)
        value = r.us_per_full_step(dt, args.steps)
        sample = r.describe(args.steps, dt)
        used = r.procs
    finally:
        r.close()
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def workload_config(w, args):
    cfg = {"workload": w.name}
    for k in ("batch", "nheads", "headdim", "dstate", "ngroups", "dk", "dv", "buf_len", "drafts"):
        if hasattr(w, k):
            cfg[k] = getattr(w, k)
    rc = getattr(w, "read_copy", False)
    rc_name = {"f16": " + fp16 read copy", "f8": " + fp8 e4m3 read copy (row scales)"}.get(rc, " + bf16 read copy")
    cfg["state"] = "fp32 checkpoint" + (rc_name if rc else "")
    cfg["io_dtype"] = "bf16 records, " + args.out_dtype + " outputs"
    cfg["l2"] = "working set larger than L2: the full checkpoint is streamed every step"
    return cfg


# ----------------------------------------------------------------------------- GPU timing

def time_calls(fn, n, stream):
    """Run fn(i) n times on `stream` with an event after each call; returns
    (total ms, per-call ms list)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    ev[0].record(stream)
    for i in range(n):
        fn(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
    return ev[0].elapsed_time(ev[n]), per


def bench_mamba2_ar(args, dist):
    import torch

    from recurrent_state_decode_gb300 import binding as bd
    from recurrent_state_decode_gb300 import bytes_model as bm
    from recurrent_state_decode_gb300 import inputs as I
    from recurrent_state_decode_gb300.state import mamba2_from_workload

    w = I.WORKLOADS[args.workload]
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    out = bd.RSSM_BF16 if args.out_dtype == "bf16" else bd.RSSM_F32
    out_bytes = 2 if out == bd.RSSM_BF16 else 4
    st, A, D, _, _, counts0 = mamba2_from_workload(w, dev, out)
    W_, K = args.warmup, args.steps
    recs = [I.mamba2_step_inputs(w, t, dev) for t in range(W_ + K)]
    y = st.new_output()
    stream = torch.cuda.current_stream(dev)
    # the shape-specialised step advances the cursors itself; the generic one
    # is followed by the cursor kernel
    fast = w.dstate == 128 and w.headdim % 64 == 0 and w.buf_len <= 31
    launches_per_step = 1 if fast else 2

    if args.mode == "profile":
        for t in range(W_ + K):
            st.step(recs[t], A, D, y)
        torch.cuda.synchronize()
        c0 = counts0.cpu().tolist()
        write_bytes(args, [bm.mamba2_step_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len,
                                                [(c + t) % w.buf_len for c in c0], w.read_copy, out_bytes)
                           for t in range(W_ + K)])
        return None

    # --- ReplaySSM step
    for t in range(W_):
        st.step(recs[t], A, D, y)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    total_ms, per = time_calls(lambda i: st.step(recs[W_ + i], A, D, y), K, stream)
    clk = clocks.stop()
    dist.barrier()
    bd.check(int(st.status.item()), "device status")
    c0 = counts0.cpu().tolist()
    L = w.buf_len
    alg_bytes = sum(bm.mamba2_step_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, L,
                                         [(c + W_ + i) % L for c in c0], w.read_copy, out_bytes) for i in range(K))
    us_step = dist.max(total_ms * 1e3 / K)
    mean_call_ms = total_ms / K
    achieved_gbs = (alg_bytes / K) / (mean_call_ms * 1e-3) / 1e9

    # --- conventional comparator over the same steps
    conv_us, conv_gbs = time_mamba2_conventional(st, A, D, recs, W_, K, stream, dist, w, out_bytes)

    # --- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = e2e_mamba2(st, A, D, w, dev, K, W_, y.dtype)
        e2e["value"] = dist.max(e2e["value"])
    del recs, st
    torch.cuda.empty_cache()

    peak, peak_kind = measured_peak()
    tokens = dist.sum(w.batch * K) / (dist.max(total_ms) * 1e-3)
    res = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": dist.world, "steps": K, "warmup": W_,
        "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic", "config": workload_config(w, args),
        "tokens_per_s": tokens,
        "hbm_gbs": achieved_gbs,
        "conventional_us_per_step": conv_us,
        "conventional_hbm_gbs": conv_gbs,
        "speedup_vs_conventional": conv_us / us_step,
        "algorithmic_bytes_per_step": alg_bytes / K,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "peak_source": peak_kind,
                     "frac_vs_nominal": achieved_gbs / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": profiled_traffic("mamba2_step_serving.txt", KERNEL_SOURCES),
                     "kernel": "m2_step_fast_kernel (advances the cursors itself; timed per call)"},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "e2e": e2e,
    }
    if args.workload == "mamba2_serving" and dist.world == 1:
        res["workloads"] = other_workloads(args, dev, out, out_bytes, min(K, 256), W_, dist, stream)
    return res


def time_mamba2_conventional(st, A, D, recs, W_, K, stream, dist, w, out_bytes):
    import torch

    from recurrent_state_decode_gb300 import binding as bd
    from recurrent_state_decode_gb300 import bytes_model as bm
    state = st.ckpt.clone()
    yc = st.new_output()
    desc = st.desc

    def conv(i):
        r = recs[W_ + i] if i >= 0 else recs[0]
        bd.check(bd.rssm_mamba2_conventional_step(desc, state, r["x"], r["z"], r["B"], r["C"], r["dt"], A, D, yc))

    for _ in range(W_):
        conv(-1)
    torch.cuda.synchronize()
    dist.barrier()
    conv_ms, _ = time_calls(conv, K, stream)
    conv_us = dist.max(conv_ms * 1e3 / K)
    conv_bytes = bm.mamba2_conventional_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, w.batch, out_bytes)
    del state
    return conv_us, conv_bytes / (conv_us * 1e-6) / 1e9


def other_workloads(args, dev, out, out_bytes, K, W_, dist, stream):
    """The other hot-path workloads, each timed like the main one on K steps."""
    import torch

    from recurrent_state_decode_gb300 import binding as bd
    from recurrent_state_decode_gb300 import bytes_model as bm
    from recurrent_state_decode_gb300 import inputs as I
    from recurrent_state_decode_gb300.state import gdn_from_workload, kda_from_workload, mamba2_from_workload
    peak, _ = measured_peak()
    res = {}

    # bf16 and fp16 read copies of the checkpoint (non-flush steps read 2 bytes per state element)
    for name in ("mamba2_bf16_read", "mamba2_f16_read", "mamba2_f8_read"):
        w = I.WORKLOADS[name]
        st, A, D, _, _, counts0 = mamba2_from_workload(w, dev, out)
        recs = [I.mamba2_step_inputs(w, t, dev) for t in range(W_ + K)]
        y = st.new_output()
        for t in range(W_):
            st.step(recs[t], A, D, y)
        torch.cuda.synchronize()
        ms, _ = time_calls(lambda i: st.step(recs[W_ + i], A, D, y), K, stream)
        bd.check(int(st.status.item()), "device status")
        c0 = counts0.cpu().tolist()
        nbytes = sum(bm.mamba2_step_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len,
                                          [(c + W_ + i) % w.buf_len for c in c0], w.read_copy, out_bytes)
                     for i in range(K)) / K
        us = ms * 1e3 / K
        res[w.name] = {"us_per_step": us, "hbm_gbs": nbytes / (us * 1e-6) / 1e9,
                       "frac": nbytes / (us * 1e-6) / 1e9 / peak, "algorithmic_bytes_per_step": nbytes, "steps": K}
        del st, recs
        torch.cuda.empty_cache()

    # emulated read precision (e4m3, one scale per 64-row tile): the fp32 checkpoint read through a
    # quantise-dequantise on non-flush steps, the per-call error report reduced after the step
    w = I.WORKLOADS["mamba2_serving"]
    st, A, D, _, _, counts0 = mamba2_from_workload(w, dev, out)
    recs = [I.mamba2_step_inputs(w, t, dev) for t in range(W_ + K)]
    y = st.new_output()
    emu = bd.emulation(bd.RSSM_EMU_E4M3, bd.RSSM_EMU_SCALE_TILE64)
    err = torch.zeros(2, dtype=torch.float64, device=dev)
    ws = torch.empty(bd.rssm_mamba2_emulated_workspace_bytes(st.desc), dtype=torch.uint8, device=dev)
    for t in range(W_):
        st.step_emulated(recs[t], A, D, y, emu, err, ws)
    torch.cuda.synchronize()
    ms, _ = time_calls(lambda i: st.step_emulated(recs[W_ + i], A, D, y, emu, err, ws), K, stream)
    bd.check(int(st.status.item()), "device status")
    e, n = err.tolist()
    c0 = counts0.cpu().tolist()
    nbytes = sum(bm.mamba2_step_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len,
                                      [(c + W_ + i) % w.buf_len for c in c0], False, out_bytes)
                 for i in range(K)) / K
    us = ms * 1e3 / K
    res["mamba2_emu_e4m3_tile64"] = {"us_per_step": us, "hbm_gbs": nbytes / (us * 1e-6) / 1e9,
                                     "frac": nbytes / (us * 1e-6) / 1e9 / peak, "algorithmic_bytes_per_step": nbytes,
                                     "read_rel_l2": (e / n) ** 0.5 if n > 0 else None, "steps": K}
    del st, recs, ws
    torch.cuda.empty_cache()

    # speculative verify + commit, K = T + 1 records per sequence per step
    w = I.WORKLOADS["mamba2_spec"]
    st, A, D, _, _, counts0 = mamba2_from_workload(w, dev, out)
    recs = [I.mamba2_verify_inputs(w, t, dev) for t in range(W_ + K)]
    kepts = [I.accepted_kept(w, t, dev) for t in range(W_ + K)]
    y = st.new_output(w.n_new)

    def spec(i):
        st.verify(recs[i], A, D, y)
        st.commit(kepts[i])

    for t in range(W_):
        spec(t)
    torch.cuda.synchronize()
    ms, _ = time_calls(lambda i: spec(W_ + i), K, stream)
    bd.check(int(st.status.item()), "device status")
    # cursor trace on the host for the bytes model (fold when count + K > L)
    counts = counts0.cpu().tolist()
    kl = [k.cpu().tolist() for k in kepts]
    nbytes = 0
    accepted = 0
    for t in range(W_ + K):
        if t >= W_:
            nbytes += bm.mamba2_verify_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len, w.n_new, counts,
                                             False, out_bytes)
            accepted += sum(kl[t])
        counts = [(0 if c + w.n_new > w.buf_len else c) + k for c, k in zip(counts, kl[t])]
    nbytes /= K
    us = ms * 1e3 / K
    tile32 = w.nheads * w.headdim * w.dstate * 4
    conv_spec_bytes = w.batch * tile32 * (1 + w.drafts)  # one state read + T snapshot writes per verify
    res[w.name] = {"us_per_step": us, "accepted_tokens_per_s": accepted / (ms * 1e-3),
                   "hbm_gbs": nbytes / (us * 1e-6) / 1e9, "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                   "algorithmic_bytes_per_step": nbytes,
                   "conventional_snapshot_bytes_per_step": conv_spec_bytes,
                   "bytes_ratio_vs_snapshot_spec": conv_spec_bytes / nbytes, "steps": K}
    del st, recs, kepts
    torch.cuda.empty_cache()

    # Gated DeltaNet AR step vs its conventional kernel
    w = I.WORKLOADS["gdn_serving"]
    st, _, _, counts0 = gdn_from_workload(w, dev, out)
    recs = [I.gdn_step_inputs(w, t, dev) for t in range(W_ + K)]
    o = st.new_output()
    for t in range(W_):
        st.step(recs[t], o)
    torch.cuda.synchronize()
    ms, _ = time_calls(lambda i: st.step(recs[W_ + i], o), K, stream)
    bd.check(int(st.status.item()), "device status")
    c0 = counts0.cpu().tolist()
    nbytes = sum(bm.gdn_step_bytes(w.nheads, w.dk, w.dv, w.buf_len, [(c + W_ + i) % w.buf_len for c in c0],
                                   out_bytes) for i in range(K)) / K
    us = ms * 1e3 / K
    S = st.S.clone()
    oc = st.new_output()

    def conv(i):
        r = recs[W_ + i]
        bd.check(bd.rssm_gdn_conventional_step(st.desc, S, r["q"], r["k"], r["v"], r["g"], r["beta"], oc))

    conv(0)
    torch.cuda.synchronize()
    cms, _ = time_calls(conv, K, stream)
    cus = cms * 1e3 / K
    cbytes = bm.gdn_conventional_bytes(w.nheads, w.dk, w.dv, w.batch, out_bytes)
    res[w.name] = {"us_per_step": us, "hbm_gbs": nbytes / (us * 1e-6) / 1e9, "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                   "algorithmic_bytes_per_step": nbytes, "conventional_us_per_step": cus,
                   "conventional_hbm_gbs": cbytes / (cus * 1e-6) / 1e9, "speedup_vs_conventional": cus / us,
                   "steps": K}
    del st, recs, S
    torch.cuda.empty_cache()

    # Kimi Delta Attention AR step vs its conventional kernel
    w = I.WORKLOADS["kda_serving"]
    st, _, _, counts0 = kda_from_workload(w, dev, out)
    recs = [I.kda_step_inputs(w, t, dev) for t in range(W_ + K)]
    o = st.new_output()
    for t in range(W_):
        st.step(recs[t], o)
    torch.cuda.synchronize()
    ms, _ = time_calls(lambda i: st.step(recs[W_ + i], o), K, stream)
    bd.check(int(st.status.item()), "device status")
    c0 = counts0.cpu().tolist()
    nbytes = sum(bm.kda_step_bytes(w.nheads, w.dk, w.dv, w.buf_len, [(c + W_ + i) % w.buf_len for c in c0],
                                   out_bytes) for i in range(K)) / K
    us = ms * 1e3 / K
    S = st.S.clone()
    oc = st.new_output()

    def kconv(i):
        r = recs[W_ + i]
        bd.check(bd.rssm_kda_conventional_step(st.desc, S, r["q"], r["k"], r["v"], r["g"], r["beta"], oc))

    kconv(0)
    torch.cuda.synchronize()
    cms, _ = time_calls(kconv, K, stream)
    cus = cms * 1e3 / K
    cbytes = bm.kda_conventional_bytes(w.nheads, w.dk, w.dv, w.batch, out_bytes)
    res[w.name] = {"us_per_step": us, "hbm_gbs": nbytes / (us * 1e-6) / 1e9, "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                   "algorithmic_bytes_per_step": nbytes, "conventional_us_per_step": cus,
                   "conventional_hbm_gbs": cbytes / (cus * 1e-6) / 1e9, "speedup_vs_conventional": cus / us,
                   "steps": K}
    del st, recs, S
    torch.cuda.empty_cache()

    # Gated DeltaNet speculative verify + commit, K = T + 1 records per sequence per step
    w = I.WORKLOADS["gdn_spec"]
    st, _, _, counts0 = gdn_from_workload(w, dev, out)
    recs = [I.gdn_verify_inputs(w, t, dev) for t in range(W_ + K)]
    kepts = [I.accepted_kept(w, t, dev) for t in range(W_ + K)]
    o = st.new_verify_output(w.n_new)

    def gspec(i):
        st.verify(recs[i], o)
        st.commit(kepts[i])

    for t in range(W_):
        gspec(t)
    torch.cuda.synchronize()
    ms, _ = time_calls(lambda i: gspec(W_ + i), K, stream)
    bd.check(int(st.status.item()), "device status")
    counts = counts0.cpu().tolist()
    kl = [k.cpu().tolist() for k in kepts]
    nbytes = 0
    accepted = 0
    for t in range(W_ + K):
        if t >= W_:
            nbytes += bm.gdn_verify_bytes(w.nheads, w.dk, w.dv, w.buf_len, w.n_new, counts, out_bytes)
            accepted += sum(kl[t])
        counts = [(0 if c + w.n_new > w.buf_len else c) + k for c, k in zip(counts, kl[t])]
    nbytes /= K
    us = ms * 1e3 / K
    tile = w.nheads * w.dv * w.dk * 4
    conv_spec_bytes = w.batch * tile * (1 + w.drafts)  # one state read + T snapshot writes per verify
    res[w.name] = {"us_per_step": us, "accepted_tokens_per_s": accepted / (ms * 1e-3),
                   "hbm_gbs": nbytes / (us * 1e-6) / 1e9, "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                   "algorithmic_bytes_per_step": nbytes,
                   "conventional_snapshot_bytes_per_step": conv_spec_bytes,
                   "bytes_ratio_vs_snapshot_spec": conv_spec_bytes / nbytes, "steps": K}
    del st, recs, kepts
    torch.cuda.empty_cache()

    # Kimi Delta Attention speculative verify + commit, K = T + 1 records per sequence per step
    w = I.WORKLOADS["kda_spec"]
    st, _, _, counts0 = kda_from_workload(w, dev, out)
    recs = [I.kda_verify_inputs(w, t, dev) for t in range(W_ + K)]
    kepts = [I.accepted_kept(w, t, dev) for t in range(W_ + K)]
    o = st.new_verify_output(w.n_new)

    def kspec(i):
        st.verify(recs[i], o)
        st.commit(kepts[i])

    for t in range(W_):
        kspec(t)
    torch.cuda.synchronize()
    ms, _ = time_calls(lambda i: kspec(W_ + i), K, stream)
    bd.check(int(st.status.item()), "device status")
    counts = counts0.cpu().tolist()
    kl = [k.cpu().tolist() for k in kepts]
    nbytes = 0
    accepted = 0
    for t in range(W_ + K):
        if t >= W_:
            nbytes += bm.kda_verify_bytes(w.nheads, w.dk, w.dv, w.buf_len, w.n_new, counts, out_bytes)
            accepted += sum(kl[t])
        counts = [(0 if c + w.n_new > w.buf_len else c) + k for c, k in zip(counts, kl[t])]
    nbytes /= K
    us = ms * 1e3 / K
    tile = w.nheads * w.dv * w.dk * 4
    conv_spec_bytes = w.batch * tile * (1 + w.drafts)  # one state read + T snapshot writes per verify
    res[w.name] = {"us_per_step": us, "accepted_tokens_per_s": accepted / (ms * 1e-3),
                   "hbm_gbs": nbytes / (us * 1e-6) / 1e9, "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                   "algorithmic_bytes_per_step": nbytes,
                   "conventional_snapshot_bytes_per_step": conv_spec_bytes,
                   "bytes_ratio_vs_snapshot_spec": conv_spec_bytes / nbytes, "steps": K}
    del st, recs, kepts
    torch.cuda.empty_cache()
    return res


def e2e_mamba2(st, A, D, w, dev, K, W_, y_dtype):
    """µs/step through rssm_mamba2_step with each step's record copied from pinned
    host memory and its output copied back, pipelined on two copy streams."""
    import torch

    from recurrent_state_decode_gb300 import inputs as I
    pool = 8
    host = []
    for t in range(pool):
        r = I.mamba2_step_inputs(w, 10_000 + t, dev)
        host.append({k: v.cpu().pin_memory() for k, v in r.items()})
    dbuf = [{k: torch.empty_like(v, device=dev) for k, v in host[0].items()} for _ in range(2)]
    ybuf = [st.new_output() for _ in range(2)]
    yhost = torch.empty(ybuf[0].shape, dtype=y_dtype).pin_memory()
    comp = torch.cuda.current_stream(dev)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    loaded = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    h2d_bytes = sum(v.numel() * v.element_size() for v in host[0].values())
    d2h_bytes = ybuf[0].numel() * ybuf[0].element_size()

    def one(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(done[b])
            for k, v in host[i % pool].items():
                dbuf[b][k].copy_(v, non_blocking=True)
            loaded[b].record(h2d)
        comp.wait_event(loaded[b])
        if i >= 2:
            comp.wait_event(copied[b])
        st.step(dbuf[b], A, D, ybuf[b], stream=comp.cuda_stream)
        done[b].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(done[b])
            yhost.copy_(ybuf[b], non_blocking=True)
            copied[b].record(d2h)

    for i in range(W_):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        one(i)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    return {"value": dt * 1e6 / K, "unit": UNIT, "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "how": "wall clock, K pipelined steps: H2D of the record (pinned), rssm_mamba2_step, D2H of y"}


def write_bytes(args, per_call):
    """Profile mode: the algorithmic bytes of each call, in call order, for the ncu summaries."""
    if args.bytes_out:
        with open(args.bytes_out, "w") as f:
            json.dump({"workload": args.workload, "bytes_per_call": per_call}, f)


def spec_bytes(fn, w, counts0, kepts, out_bytes, n):
    """Algorithmic bytes of n verifies from initial counts (fold when count + K > L)."""
    counts = counts0.cpu().tolist()
    out = []
    for t in range(n):
        out.append(fn(counts))
        kl = kepts[t].cpu().tolist()
        counts = [(0 if c + w.n_new > w.buf_len else c) + k for c, k in zip(counts, kl)]
    return out


def profile_other(args, dist):
    """A few calls of the speculative, delta-rule or emulated-read workload, untimed (for ncu)."""
    import torch

    from recurrent_state_decode_gb300 import binding as bd
    from recurrent_state_decode_gb300 import inputs as I
    from recurrent_state_decode_gb300.state import gdn_from_workload, kda_from_workload, mamba2_from_workload
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    out = bd.RSSM_BF16 if args.out_dtype == "bf16" else bd.RSSM_F32
    w = I.WORKLOADS["mamba2_serving" if args.workload == "mamba2_emu_e4m3_tile64" else args.workload]
    n = args.warmup + args.steps
    from recurrent_state_decode_gb300 import bytes_model as bm
    ob = 2 if out == bd.RSSM_BF16 else 4
    kepts = [I.accepted_kept(w, t, dev) for t in range(n)] if getattr(w, "drafts", 0) else None
    if args.workload == "mamba2_emu_e4m3_tile64":
        st, A, D, _, _, counts0 = mamba2_from_workload(w, dev, out)
        y = st.new_output()
        err = torch.zeros(2, dtype=torch.float64, device=dev)
        ws = torch.empty(bd.rssm_mamba2_emulated_workspace_bytes(st.desc), dtype=torch.uint8, device=dev)
        emu = bd.emulation(bd.RSSM_EMU_E4M3, bd.RSSM_EMU_SCALE_TILE64)
        for t in range(n):
            st.step_emulated(I.mamba2_step_inputs(w, t, dev), A, D, y, emu, err, ws)
        c0 = counts0.cpu().tolist()
        per = [bm.mamba2_step_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len,
                                    [(c + t) % w.buf_len for c in c0], False, ob) for t in range(n)]
    elif args.workload == "gdn_serving":
        st, _, _, counts0 = gdn_from_workload(w, dev, out)
        o = st.new_output()
        for t in range(n):
            st.step(I.gdn_step_inputs(w, t, dev), o)
        c0 = counts0.cpu().tolist()
        per = [bm.gdn_step_bytes(w.nheads, w.dk, w.dv, w.buf_len, [(c + t) % w.buf_len for c in c0], ob)
               for t in range(n)]
    elif args.workload == "kda_serving":
        st, _, _, counts0 = kda_from_workload(w, dev, out)
        o = st.new_output()
        for t in range(n):
            st.step(I.kda_step_inputs(w, t, dev), o)
        c0 = counts0.cpu().tolist()
        per = [bm.kda_step_bytes(w.nheads, w.dk, w.dv, w.buf_len, [(c + t) % w.buf_len for c in c0], ob)
               for t in range(n)]
    elif args.workload == "kda_spec":
        st, _, _, counts0 = kda_from_workload(w, dev, out)
        o = st.new_verify_output(w.n_new)
        for t in range(n):
            st.verify(I.kda_verify_inputs(w, t, dev), o)
            st.commit(kepts[t])
        per = spec_bytes(lambda c: bm.kda_verify_bytes(w.nheads, w.dk, w.dv, w.buf_len, w.n_new, c, ob),
                         w, counts0, kepts, ob, n)
    elif args.workload == "gdn_spec":
        st, _, _, counts0 = gdn_from_workload(w, dev, out)
        o = st.new_verify_output(w.n_new)
        for t in range(n):
            st.verify(I.gdn_verify_inputs(w, t, dev), o)
            st.commit(kepts[t])
        per = spec_bytes(lambda c: bm.gdn_verify_bytes(w.nheads, w.dk, w.dv, w.buf_len, w.n_new, c, ob),
                         w, counts0, kepts, ob, n)
    else:
        st, A, D, _, _, counts0 = mamba2_from_workload(w, dev, out)
        y = st.new_output(w.n_new)
        for t in range(n):
            st.verify(I.mamba2_verify_inputs(w, t, dev), A, D, y)
            st.commit(kepts[t])
        per = spec_bytes(lambda c: bm.mamba2_verify_bytes(w.nheads, w.headdim, w.dstate, w.ngroups, w.buf_len,
                                                          w.n_new, c, False, ob), w, counts0, kepts, ob, n)
    torch.cuda.synchronize()
    bd.check(int(st.status.item()), "device status")
    write_bytes(args, per)
    return None


# Keys of the contract, in the order they are printed; every other key follows,
# the in-run comparison with the conventional kernel last.
CONTRACT_KEYS = ["impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data", "config", "gpu_launches", "clocks", "roofline", "e2e",
                 "cpu_baseline"]
TAIL_KEYS = ["tokens_per_s", "hbm_gbs", "algorithmic_bytes_per_step", "workloads", "conventional_us_per_step",
             "conventional_hbm_gbs", "speedup_vs_conventional"]


def _round(v, digits=4):
    if isinstance(v, float):
        return float(f"{v:.{digits}g}")
    if isinstance(v, dict):
        return {k: _round(x, digits) for k, x in v.items()}
    if isinstance(v, list):
        return [_round(x, digits) for x in v]
    return v


def compact(res):
    """The printed line: floats to 4 significant digits, each extra workload
    reduced to its time, roofline fraction and (where it has one) speedup over
    its conventional kernel, the comparison with the conventional kernel at
    the end of the line."""
    out = {k: res[k] for k in CONTRACT_KEYS if k in res}
    wl = res.get("workloads")
    if wl:
        short = {}
        for name, v in wl.items():
            e = {"us": v["us_per_step"], "frac": v["frac"]}
            if "speedup_vs_conventional" in v:
                e["conv_us"] = v["conventional_us_per_step"]
                e["speedup"] = v["speedup_vs_conventional"]
            if "accepted_tokens_per_s" in v:
                e["acc_tok_s"] = v["accepted_tokens_per_s"]
            if v.get("read_rel_l2") is not None:
                e["read_rel_l2"] = v["read_rel_l2"]
            short[name] = e
        res = dict(res, workloads=short)
    for k in list(res):
        if k not in out and k not in TAIL_KEYS:
            out[k] = res[k]
    for k in TAIL_KEYS:
        if k in res:
            out[k] = res[k]
    return _round(out)


def main(argv=None):
    args = parse(argv)
    dist = Dist()
    try:
        if args.impl == "reference":
            res = run_reference(args, dist)
        else:
            from recurrent_state_decode_gb300 import binding
            binding.load()
            if args.mode == "profile" and args.workload in ("gdn_serving", "mamba2_spec", "gdn_spec", "kda_serving",
                                                            "kda_spec", "mamba2_emu_e4m3_tile64"):
                res = profile_other(args, dist)
            elif args.workload.startswith("mamba2") and "spec" not in args.workload:
                res = bench_mamba2_ar(args, dist)
            else:
                raise SystemExit(f"workload {args.workload}: run it with --mode profile, or read the "
                                 "'workloads' object of the default run")
            if res is not None and dist.rank == 0 and not args.no_cpu_baseline and dist.world == 1:
                res["cpu_baseline"] = cpu_baselines(args.workload, args.cpu_seconds)
        if res is not None and dist.rank == 0:
            if args.detail:
                with open(args.detail, "w") as f:
                    json.dump(res, f, indent=1)
            print(json.dumps(compact(res)), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
