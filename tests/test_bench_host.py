"""Host-side helpers of bench.py that need no GPU: the roofline traffic lookup
in a committed ncu summary (used only while the summary's source hash matches
the kernel file) and the whole-job aggregation at one rank."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _fake_tree(tmp_path, src: bytes, summary_sha: str, traffic="123456789"):
    csrc = tmp_path / "two_compressed_kv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k_fake.cu").write_bytes(src)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "fake.txt").write_text(
        f"kernel: fake\nkernel_source_sha256: {summary_sha}\n"
        f"dram_bytes_per_launch_full_size: {traffic}\n")


def test_traffic_is_read_only_for_the_captured_source(tmp_path, monkeypatch):
    src = b"__global__ void k() {}\n"
    _fake_tree(tmp_path, src, hashlib.sha256(src).hexdigest())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("k_fake.cu", "fake.txt") == pytest.approx(123456789.0)
    # the kernel changed after the capture: no traffic figure
    (tmp_path / "two_compressed_kv_gb300" / "csrc" / "k_fake.cu").write_bytes(src + b"// edit\n")
    assert bench.committed_traffic("k_fake.cu", "fake.txt") is None
    assert bench.committed_traffic("k_fake.cu", "missing.txt") is None


def test_traffic_rejects_a_malformed_summary(tmp_path, monkeypatch):
    src = b"x"
    _fake_tree(tmp_path, src, hashlib.sha256(src).hexdigest(), traffic="n/a")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("k_fake.cu", "fake.txt") is None


def test_committed_score_summary_names_its_source_and_traffic():
    path = os.path.join(ROOT, "profiles", "score_kernel_headline_128k.txt")
    text = open(path).read()
    assert "kernel_source_sha256:" in text and "dram_bytes_per_launch_full_size:" in text
    assert "ncu --clock-control none" in text or "ncu --set full --clock-control none" in text


def test_job_value_single_rank():
    ms_step, value = bench._job_value(80.0, 10, 4.0e6, 1, "cpu")
    assert ms_step == pytest.approx(8.0)
    assert value == pytest.approx(4.0e6 / 8e-3)


def test_oracle_sample_prepares_once_and_times_decodes():
    from two_compressed_kv_gb300 import workloads as W
    w = W.small_workload("bench-sample", ctx=256, top_k=16)
    prep = bench.oracle_prepare(w)
    assert prep["T"] == 256 and prep["q"].shape == (w.group, 128)
    value, reps, per = bench.oracle_decode_sample(w, 0.05, prep)
    assert reps >= 1 and per > 0 and value == pytest.approx(256 / (per * w.n_kv_heads))


def test_host_cpu_description():
    info = bench.host_cpu()
    assert info["cpu_count"] >= 1 and isinstance(info["cpu_model"], str)
