"""Host logic of bench.py that needs no GPU: the job rate over ranks, the row
blocks of a split batch, and the roofline traffic taken from the committed
ncu capture only while it matches the kernel sources."""

import json

import pytest

import bench


def test_job_rate_counts_every_rank():
    assert bench.job_rate(256, 1, 1e-5) == pytest.approx(256 / 1e-5)
    assert bench.job_rate(256, 4, 2e-5) == pytest.approx(4 * 256 / 2e-5)


def test_row_block_of_the_bench_split():
    # N ranks of 256 rows each: rank r starts at row 256 r
    assert [bench.row_block(4 * 256, r, 4) for r in range(4)] == [(0, 256), (256, 512), (512, 768), (768, 1024)]
    assert bench.row_block(256, 0, 1) == (0, 256)


def test_profiled_traffic_follows_the_source_hash(monkeypatch, tmp_path):
    path = tmp_path / "capture.json"
    path.write_text(json.dumps({"kernel": "sample_kernel", "dram_bytes_per_launch": 65_800_000,
                                "source_sha": "abcdabcdabcdabcd", "command": "ncu ..."}))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "abcdabcdabcdabcd")
    assert bench.profiled_traffic(str(path)) == 65_800_000.0
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0000000000000000")
    assert bench.profiled_traffic(str(path)) is None            # a changed kernel has no counters
    assert bench.profiled_traffic(str(tmp_path / "missing.json")) is None


def test_committed_capture_is_machine_readable():
    with open(bench.PROFILE_JSON) as fh:
        data = json.load(fh)
    assert data["kernel"] == "sample_kernel" and data["dram_bytes_per_launch"] > 65e6
    assert len(data["source_sha"]) == 16 and data["command"].startswith("ncu ")


def test_measured_peaks_has_a_copy_rate():
    peak, kind = bench.measured_peaks()
    assert peak > 1000.0 and kind in ("measured", "fallback")
