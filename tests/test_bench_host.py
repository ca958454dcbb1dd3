"""bench.py host logic without a GPU: the committed DRAM-traffic captures are used only for the sources
they were taken on, flop counts and peaks are read as documented."""

import json
import os

import pytest

import bench


def test_traffic_capture_follows_its_sources():
    """Each committed capture names its kernel's sources; bench reports its bytes while their digest
    matches the tree and null once a source has changed since the capture."""
    for workload, (fname, files) in bench.TRAFFIC.items():
        path = os.path.join(bench.ROOT, "profiles", fname)
        if not os.path.exists(path):
            continue
        with open(path) as fh:
            rec = json.load(fh)
        assert [os.path.basename(p) for p in rec["sources"]] == list(files)
        current = rec["kernel_source_sha256"] == bench.source_digest(files)
        want = rec["per_launch_bytes"][f"{workload}/gram"] if current else None
        assert bench.measured_traffic(workload, "gram") == want


def test_traffic_is_none_for_other_workloads_and_forms():
    assert bench.measured_traffic("no-such-workload", "gram") is None
    assert bench.measured_traffic("llama3-8b-muon-set", "direct") is None


def test_stale_digest_hides_the_capture(tmp_path, monkeypatch):
    """A capture taken on other sources is not reported."""
    fname, files = bench.TRAFFIC["small-set-2560"]
    src = os.path.join(bench.ROOT, "profiles", fname)
    if not os.path.exists(src):
        pytest.skip("no committed capture")
    with open(src) as f:
        rec = json.load(f)
    rec["kernel_source_sha256"] = "0" * 64
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / fname).write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda files: "1" * 64)
    assert bench.measured_traffic("small-set-2560", "gram") is None


def test_total_flops_counts_every_matrix():
    import newton_schulz_momentum_gb300 as dm
    shapes = [("a", 128, 512), ("b", 512, 128), ("c", 4096, 4096)]
    assert bench.total_flops(shapes, "gram") == sum(dm.gram_flops(r, c) for _, r, c in shapes)
    assert bench.total_flops(shapes, "direct") == sum(dm.direct_flops(r, c) for _, r, c in shapes)
    auto = bench.total_flops(shapes, "auto")
    assert auto == dm.gram_flops(128, 512) + dm.gram_flops(512, 128) + dm.direct_flops(4096, 4096)


def test_peaks_read_the_measured_file_or_fall_back():
    hbm, burst, sustained, src = bench.peaks()
    assert src in ("measured", "fallback")
    assert hbm > 0 and burst >= sustained > 0
