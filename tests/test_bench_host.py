"""CPU tests of bench.py's host logic: multi-rank coordination over gloo
(world size 2, replicas: max/sum over ranks, rank-0 output only) and the
algorithmic bytes model."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from recurrent_state_decode_gb300 import bytes_model as bm


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    d = bench.Dist()
    try:
        d.barrier()
        q.put((rank, d.max(10.0 + rank), d.sum(1.0 + rank)))
    finally:
        d.close()


def test_dist_max_sum_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0, 3.0), (1, 11.0, 3.0)]


def test_reference_arm_other_ranks_exit(monkeypatch):
    class Fake:
        rank = 1
    assert bench.run_reference(bench.parse(["--impl", "reference"]), Fake()) is None


def test_bytes_model_serving_cycle():
    """Average over a full L-cycle of staggered windows at the serving shape:
    4 MiB read every step, 4 MiB written on 1 step in 16, 2 x 37,376 B of
    record in + append on the 15 non-flush steps (one read on the flush),
    7.5 window records of 18,944 B on average, 16,384 B of bf16 y, 32 B of cursor."""
    H, P, N, G, L = 128, 64, 128, 8, 16
    per_seq = sum(bm.mamba2_step_bytes(H, P, N, G, L, [c]) for c in range(L)) / L
    expect = 4194304 + 4194304 / 16 + (15 * 2 * 37376 + 37376) / 16 + 7.5 * 18944 + 16384 + 32
    assert per_seq == pytest.approx(expect)
    conv = bm.mamba2_conventional_bytes(H, P, N, G, 1)
    assert conv == 2 * 4194304 + 37376 + 16384
    # GDN serving shape: 2 MiB state per sequence; a past record is read back as
    # k, g and its cached correction e (dv fp32), and an append stores e too
    g = sum(bm.gdn_step_bytes(32, 128, 128, 16, [c]) for c in range(16)) / 16
    rec = 32 * (2 * 256 + 256 + 8)
    e = 32 * 512
    past = 32 * (256 + 4) + e
    assert g == pytest.approx(2097152 * 17 / 16 + (15 * (2 * rec + e) + rec) / 16 + 7.5 * past + 32 * 128 * 2 + 32)
    # GDN verify, K = 4: a fold on count 13 (13 + 4 > 16), none on count 12
    v = bm.gdn_verify_bytes(32, 128, 128, 16, 4, [12, 13])
    assert v == (2097152 + 4 * (2 * rec + e) + 12 * past + 4 * 32 * 128 * 2 + 68) + \
        (2 * 2097152 + 4 * (2 * rec + e) + 13 * past + 4 * 32 * 128 * 2 + 68)
    # KDA serving shape: as GDN, with g one fp32 per key channel in the record and past records
    kd = sum(bm.kda_step_bytes(32, 128, 128, 16, [c]) for c in range(16)) / 16
    krec = 32 * (2 * 256 + 256 + 512 + 4)
    kpast = 32 * (256 + 512) + e
    assert kd == pytest.approx(2097152 * 17 / 16 + (15 * (2 * krec + e) + krec) / 16 + 7.5 * kpast + 32 * 128 * 2 + 32)
    assert bm.kda_conventional_bytes(32, 128, 128, 2) == 2 * (2 * 2097152 + krec + 32 * 128 * 2)
    kv = bm.kda_verify_bytes(32, 128, 128, 16, 4, [12, 13])
    assert kv == (2097152 + 4 * (2 * krec + e) + 12 * kpast + 4 * 32 * 128 * 2 + 68) + \
        (2 * 2097152 + 4 * (2 * krec + e) + 13 * kpast + 4 * 32 * 128 * 2 + 68)


def test_oracle_baseline_runs_on_several_cores():
    """The CPU baseline's worker pool (spawned processes, one chunk of
    sequences each) times the oracle on the tiny configuration."""
    v, sample, used = bench.oracle_baseline("mamba2_tiny", 0.2, 2)
    assert v > 0 and used == 2
    assert "4 of 4 sequences on 2 worker processes" in sample


def test_printed_line_keeps_the_claims_in_its_tail():
    """The contract's keys come first; the comparison with the conventional
    kernel closes the line, which stays short enough to be read whole."""
    wl = {n: {"us_per_step": 123.456789, "frac": 0.612345, "speedup_vs_conventional": 1.3456,
              "conventional_us_per_step": 188.0123, "accepted_tokens_per_s": 3.0e6, "hbm_gbs": 4600.1,
              "algorithmic_bytes_per_step": 6.4e8, "steps": 20}
          for n in ("mamba2_bf16_read", "mamba2_f16_read", "mamba2_f8_read", "mamba2_spec", "gdn_serving",
                    "kda_serving", "gdn_spec", "kda_spec", "mamba2_emu_e4m3")}
    res = {"metric": bench.METRIC, "value": 209.1234567, "unit": bench.UNIT, "n_gpus": 1, "steps": 20, "warmup": 5,
           "ms_per_step": 0.2091234, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
           "dtype": "f32", "data": "synthetic", "config": {"workload": "mamba2_serving"}, "workloads": wl,
           "speedup_vs_conventional": 1.5432, "conventional_us_per_step": 322.8, "tokens_per_s": 1.2e6,
           "cpu_baseline": {"value": 1.0, "per_config": {c: {"value": 1.0, "cores": 16} for c in bench.CPU_CONFIGS}}}
    line = __import__("json").dumps(bench.compact(res))
    keys = list(bench.compact(res))
    assert keys[:3] == ["metric", "value", "unit"] and keys[-1] == "speedup_vs_conventional"
    assert line.index('"cpu_baseline"') < line.index('"workloads"')
    assert len(line[line.index('"workloads"'):]) < 1500
