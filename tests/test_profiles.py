"""The committed ncu summaries against the bytes model: each kernel's measured
DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) is
within a few percent of the algorithmic bytes the model counts, so no kernel
re-reads what it should read once. CPU only: the summaries are text."""
import glob
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARIES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.txt")))


def _fields(path):
    out = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


def test_there_are_kernel_summaries():
    names = {os.path.basename(p) for p in SUMMARIES}
    assert {"mamba2_step_serving.txt", "mamba2_step_bf16_read.txt", "mamba2_step_emulated_e4m3.txt",
            "mamba2_verify_spec.txt", "gdn_step_serving.txt", "gdn_verify_spec.txt", "kda_step_serving.txt",
            "kda_verify_spec.txt"} <= names


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_summary_was_taken_on_the_committed_sources(path):
    """A summary's source hash is that of the kernel sources as they are now
    (the hash bench.py checks before quoting a summary's DRAM traffic): a
    change to a kernel makes its summary stale until it is captured again."""
    import bench
    f = _fields(path)
    assert f["source_sha256"] == bench.source_hash(f["source_files"].split()), "recapture this summary"


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_dram_traffic_matches_the_bytes_model(path):
    f = _fields(path)
    dram, alg = float(f["dram_bytes_per_launch"]), float(f["algorithmic_bytes_per_launch"])
    assert 0.95 <= dram / alg <= 1.15, (dram, alg)
    assert abs(float(f["dram_over_algorithmic"]) - dram / alg) < 5e-3


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_summary_names_its_command_and_sources(path):
    f = _fields(path)
    assert f["command"].startswith("ncu ") and "--clock-control none" in f["command"]
    assert "python bench.py" in f["command"]
    for src in f["source_files"].split():
        assert os.path.exists(os.path.join(ROOT, src)), src
