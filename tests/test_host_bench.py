"""Host logic of bench.py that decides what the bench line reports: a DRAM
traffic figure is taken from a committed ncu summary only while the summary's
recorded source hash matches the kernel's current sources."""
import os

import bench


def write_summary(tmp_path, tag, workload, sha, dram="123456", note=""):
    d = tmp_path / "profiles"
    d.mkdir(exist_ok=True)
    (d / f"{tag}_{workload}.md").write_text(
        "# summary\n\n"
        f"- dram_bytes_per_launch: {dram}\n"
        f"- kernel_sources_sha256: `{sha}`{note}\n")


def test_traffic_read_while_hash_matches(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    real = os.path.dirname(os.path.abspath(bench.__file__))
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda tag: "abc123" if tag == "decode_nvfp4" else "zzz")
    write_summary(tmp_path, "decode_nvfp4", "w1", "abc123", note=" (the decode step's source set)")
    assert bench.profiled_traffic("decode_nvfp4", "w1") == 123456.0
    write_summary(tmp_path, "decode_nvfp4", "w2", "abc124")
    assert bench.profiled_traffic("decode_nvfp4", "w2") is None           # stale summary
    assert bench.profiled_traffic("decode_nvfp4", "missing") is None
    write_summary(tmp_path, "decode_nvfp4", "w3", "abc123", dram="n/a")
    assert bench.profiled_traffic("decode_nvfp4", "w3") is None
    assert os.path.isdir(real)


def test_source_hash_covers_every_listed_file():
    for tag, files in bench.KERNEL_SOURCES.items():
        h = bench.kernel_sources_hash(tag)
        assert len(h) == 16
        for f in files:
            assert os.path.exists(os.path.join(bench.ROOT, "nvfp4_quantized_paged_nvfp4kv_gb300", "csrc", f)), f
