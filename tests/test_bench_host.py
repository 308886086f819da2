"""Host logic of bench.py that needs no GPU: the job rate over ranks and the
roofline traffic taken from the committed ncu summary only while it matches
the kernel sources."""

import pytest

import bench


def test_job_rate_counts_every_rank():
    assert bench.job_rate(256, 1, 1e-5) == pytest.approx(256 / 1e-5)
    assert bench.job_rate(256, 4, 2e-5) == pytest.approx(4 * 256 / 2e-5)


def _summary_sha():
    with open(bench.PROFILE_SUMMARY) as fh:
        for line in fh:
            if line.startswith("- source_sha:"):
                return line.split(":", 1)[1].strip().strip("`")
    return None


def test_profiled_traffic_follows_the_source_hash(monkeypatch):
    sha = _summary_sha()
    assert sha is not None
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: sha)
    value = bench.profiled_traffic()
    assert value is not None and value > 65e6          # DRAM bytes of one launch
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0000000000000000")
    assert bench.profiled_traffic() is None            # a changed kernel has no counters


def test_measured_peaks_has_a_copy_rate():
    peak, kind = bench.measured_peaks()
    assert peak > 1000.0 and kind in ("measured", "fallback")
