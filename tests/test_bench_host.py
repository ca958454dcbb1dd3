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
    """value counts Gram as 6 m^2 n + 20 m^3 (S = (aI+Z) R a full product); as_executed as the library
    computes it, 6 m^2 n + 17 m^3; direct 15 m^2 n + 5 m^3 either way."""
    import newton_schulz_momentum_gb300 as dm
    shapes = [("a", 128, 512), ("b", 512, 128), ("c", 4096, 4096)]

    def alg(r, c):
        m, n = min(r, c), max(r, c)
        return 6 * m * m * n + 20 * m ** 3

    assert bench.total_flops(shapes, "gram") == sum(alg(r, c) for _, r, c in shapes)
    assert bench.total_flops(shapes, "gram", as_executed=True) == sum(dm.gram_flops(r, c) for _, r, c in shapes)
    assert bench.total_flops(shapes, "direct") == sum(dm.direct_flops(r, c) for _, r, c in shapes)
    auto = bench.total_flops(shapes, "auto")
    assert auto == alg(128, 512) + alg(512, 128) + dm.direct_flops(4096, 4096)


def test_headline_flop_total_matches_the_closed_form():
    """The whole Llama-3-8B set: 387.85 TFLOP per Gram step on the algorithmic count, 354.66 as executed."""
    import workloads
    shapes = workloads.llama3_8b_shapes(32)
    assert round(bench.total_flops(shapes, "gram") / 1e12, 2) == 387.85
    assert round(bench.total_flops(shapes, "gram", as_executed=True) / 1e12, 2) == 354.66


def test_owned_shapes_partition_the_set():
    """--owned: every matrix belongs to exactly one rank's share, and each share is what
    dmuon_assign_owners gives that rank."""
    import workloads
    shapes = workloads.llama3_8b_shapes(32)
    for world in (1, 2, 3, 8):
        shares = [bench.owned_shapes(shapes, world, r) for r in range(world)]
        names = sorted(n for share in shares for n, _, _ in share)
        assert names == sorted(n for n, _, _ in shapes)


def test_reference_extrapolation_covers_every_shape():
    """The reference arm's distinct oriented shapes and their counts add up to the workload."""
    import workloads
    shapes = workloads.llama3_8b_shapes(32)
    distinct = bench.distinct_oriented(shapes)
    assert sorted((min(r, c), max(r, c)) for r, c, _ in distinct) == [(1024, 4096), (4096, 4096), (4096, 14336)]
    assert sum(n for _, _, n in distinct) == 224
    small = [(f"m{i}", r, c) for i, (r, c) in enumerate(workloads.small_set_shapes())]
    assert [(min(r, c), max(r, c), n) for r, c, n in bench.distinct_oriented(small)] == [(128, 512, 2560)]


def test_cpu_info_names_the_host():
    info = bench.cpu_info()
    assert set(info) == {"cpu_model", "blas", "numpy"}
    assert info["numpy"]


def test_peaks_read_the_measured_file_or_fall_back():
    hbm, burst, sustained, src = bench.peaks()
    assert src in ("measured", "fallback")
    assert hbm > 0 and burst >= sustained > 0
