"""Host-side pieces of the benchmark that need no GPU: the algorithmic byte
count, the per-launch traffic read from a committed ncu summary (and
withheld once the kernel sources differ from the capture's), the peak
table's fallback."""
import os

import pytest


def test_algo_bytes_counts_codes_metadata_and_vectors():
    import bench
    # 28672 x 8192, M = 1, bf16 in and out: codes + f32 scale + u8 zero per
    # group + x + y
    N, K = 28672, 8192
    assert bench.algo_bytes(1, N, K) == N * K // 2 + 5 * N * K // 128 + 2 * K + 2 * N
    assert bench.algo_bytes(4, 16, 128, xb=4, yb=4) == 16 * 64 + 5 * 16 + 4 * 128 * 4 + 4 * 16 * 4


def test_profile_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    h = bench.sources_hash(["k.cu"])
    (tmp_path / "profiles" / "p.md").write_text(
        f"summary\ntraffic_bytes_per_launch: 123456\nsource_sha256: {h}\n")
    assert bench.profile_traffic("p.md", ["k.cu"]) == 123456.0
    src.write_text("kernel v2\n")  # the kernel changed since the capture
    assert bench.profile_traffic("p.md", ["k.cu"]) is None
    assert bench.profile_traffic("missing.md", ["k.cu"]) is None


def test_peaks_fall_back_without_measurements(tmp_path, monkeypatch):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.peaks()
    assert pk["source"] == "fallback" and pk["hbm_gbs"] > 0 and pk["bf16_tflops"] > 0


def test_committed_summaries_name_their_numbers():
    """Every committed profile summary that feeds the benchmark carries the
    fields the benchmark reads."""
    import bench
    text = open(os.path.join(bench.ROOT, "profiles", "gemv_decode70b_M1.md")).read()
    assert "traffic_bytes_per_launch:" in text and "source_sha256:" in text
