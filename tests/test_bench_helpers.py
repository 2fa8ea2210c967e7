"""Host-side helpers of bench.py: the end-to-end chunk rule, the gate that
keeps a stale ncu summary's traffic out of the bench line, the measured-peak
reading and the algorithmic byte count (the roofline numerator)."""

import json
import os

import pytest
import torch

import bench


def test_e2e_chunks_only_for_large_batches():
    assert bench.e2e_chunks(4096, 4096 * 131072 * 4) == 8
    assert bench.e2e_chunks(4096, (256 << 20) - 4) == 1      # below 256 MB: one chunk
    assert bench.e2e_chunks(64, 64 * 65536 * 4) == 1          # decode-sized batches
    assert bench.e2e_chunks(12, 1 << 30) == 4                 # largest of 8, 4, 2 dividing M
    assert bench.e2e_chunks(6, 1 << 30) == 2
    assert bench.e2e_chunks(7, 1 << 30) == 1
    assert bench.e2e_chunks(1, 1 << 30) == 1


def _profile(tmp_path, kernel, workload, traffic, sha):
    (tmp_path / f"{kernel}__{workload}.md").write_text(
        f"# summary\n\ntraffic_bytes_per_launch: {traffic}\nkernel_source_sha256_16: {sha}\n")


def test_profiled_traffic_needs_the_current_kernel_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    sha = bench.kernel_source_hash()
    assert len(sha) == 16
    _profile(tmp_path, "k", "w", 123456, sha)
    assert bench.profiled_traffic("k", "w") == 123456.0
    _profile(tmp_path, "k", "stale", 99, "0" * 16)              # taken on another source
    assert bench.profiled_traffic("k", "stale") is None
    assert bench.profiled_traffic("k", "missing") is None


def test_committed_summaries_parse():
    # every committed per-kernel summary carries both fields the gate reads
    for name in os.listdir(bench.PROFILES):
        if "__" not in name or name.startswith(("launches", "stream_floor")):
            continue
        text = open(os.path.join(bench.PROFILES, name)).read()
        assert "traffic_bytes_per_launch:" in text, name
        assert "kernel_source_sha256_16:" in text, name


def test_hbm_peak_reads_the_measured_file_or_falls_back(tmp_path, monkeypatch):
    f = tmp_path / "peaks.json"
    f.write_text(json.dumps({"hbm_gbs": 6769.8}))
    monkeypatch.setattr(bench, "MEASURED_PEAKS", str(f))
    v, src = bench.hbm_peak()
    assert v == 6769.8 and src.startswith("measured")
    monkeypatch.setattr(bench, "MEASURED_PEAKS", str(tmp_path / "absent.json"))
    v, src = bench.hbm_peak()
    assert v == bench.FALLBACK_HBM_GBS and src.startswith("fallback")


def test_algorithmic_bytes_counts_clamped_prefixes_and_outputs():
    ke = torch.tensor([0, 5, 100, -3, 7], dtype=torch.int32)
    N, M, K = 10, 5, 4
    # prefixes clamped to [0, N]: 0 + 5 + 10 + 0 + 7 scores, then M * K indices
    assert bench.algorithmic_bytes(ke, N, M, K) == (0 + 5 + 10 + 0 + 7) * 4 + M * K * 4
