"""Host logic of bench.py that needs no GPU: the roofline's DRAM traffic is
taken from a committed ncu summary only while that summary's recorded
source hash matches the kernel source as it stands."""
import hashlib

import bench


def _layout(tmp_path, source: bytes, profile: str):
    csrc = tmp_path / "hybrid_linear_attention_02_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_bytes(source)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(profile)


def test_traffic_read_when_the_source_matches(tmp_path, monkeypatch):
    src = b"__global__ void k() {}\n"
    sha = hashlib.sha256(src).hexdigest()
    _layout(tmp_path, src, f"# k\nsource_sha256: {sha}\ndram_bytes_per_launch: 1234500000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k.cu", "k.md") == 1234500000.0


def test_traffic_dropped_once_the_kernel_changes(tmp_path, monkeypatch):
    src = b"__global__ void k() {}\n"
    old = hashlib.sha256(b"__global__ void k() { /* the captured version */ }\n").hexdigest()
    _layout(tmp_path, src, f"source_sha256: {old}\ndram_bytes_per_launch: 1234500000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k.cu", "k.md") is None


def test_traffic_needs_both_lines_and_both_files(tmp_path, monkeypatch):
    src = b"x"
    sha = hashlib.sha256(src).hexdigest()
    _layout(tmp_path, src, f"source_sha256: {sha}\n")          # no traffic line
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k.cu", "k.md") is None
    assert bench.kernel_traffic("missing.cu", "k.md") is None
    assert bench.kernel_traffic("k.cu", "missing.md") is None


def test_job_throughput_counts_every_rank_against_the_slowest():
    # 4 ranks x 8192 tokens in 2 ms (the max over ranks) -> 16.384 M tokens/s.
    assert abs(bench.job_throughput(4, 8192, 2.0) - 16.384e6) < 1e-3
