"""Host-side rules of bench.py that need no GPU: DRAM traffic is taken from
an ncu summary only while that summary's kernel-source hash matches the
sources as they are now."""
import bench


def _write(root, workload, text):
    d = root / "profiles"
    d.mkdir(exist_ok=True)
    (d / f"decode_{workload}.md").write_text(text)


def test_traffic_only_from_a_profile_of_the_current_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0123456789abcdef")
    assert bench.profiled_traffic("w") is None  # no summary
    _write(tmp_path, "w", "kernel_source_sha256_16: 0123456789abcdef\ndram_bytes_per_launch: 3.5e8\n")
    assert bench.profiled_traffic("w") == 3.5e8
    _write(tmp_path, "w", "kernel_source_sha256_16: fedcba9876543210\ndram_bytes_per_launch: 3.5e8\n")
    assert bench.profiled_traffic("w") is None  # taken on other sources
    _write(tmp_path, "w", "kernel_source_sha256_16: 0123456789abcdef\n")
    assert bench.profiled_traffic("w") is None  # no byte count


def test_kernel_hash_follows_every_source(tmp_path, monkeypatch):
    for name in bench.KERNEL_SOURCES:
        p = tmp_path / name
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text("x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_hash()
    for name in bench.KERNEL_SOURCES:
        (tmp_path / name).write_text("y")
        h1 = bench.kernel_hash()
        assert h1 != h0
        h0 = h1
