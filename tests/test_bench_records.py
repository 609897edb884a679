"""Host-side pieces of bench.py that need no GPU: the DRAM-traffic record is
read only while every source file it lists is unchanged (otherwise
roofline.traffic is null)."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write_tree(tmp, kernel: str, sources: dict, listed: str, sha: str, value: str):
    os.makedirs(os.path.join(tmp, "profiles"))
    csrc = os.path.join(tmp, "quantized_paged_kv_q8_gb300", "csrc")
    os.makedirs(csrc)
    for name, text in sources.items():
        with open(os.path.join(csrc, name), "w") as f:
            f.write(text)
    with open(os.path.join(tmp, "profiles", f"{kernel}_dram.txt"), "w") as f:
        f.write(f"# comment: with a colon\nsource: {listed}\nsource_sha256_16: {sha}\n"
                f"dram_bytes_per_launch: {value}\n")


def test_traffic_record_follows_its_sources(tmp_path, monkeypatch):
    src = {"a.cu": "kernel a\n", "b.cuh": "header b\n"}
    sha = hashlib.sha256((src["a.cu"] + src["b.cuh"]).encode()).hexdigest()[:16]
    _write_tree(str(tmp_path), "k", src, "a.cu b.cuh", sha, "12345")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k") == 12345.0
    assert bench.traffic_record("missing") is None
    with open(tmp_path / "quantized_paged_kv_q8_gb300" / "csrc" / "b.cuh", "a") as f:
        f.write("// edited\n")                      # any listed file changing voids the record
    assert bench.traffic_record("k") is None


def test_traffic_record_rejects_bad_records(tmp_path, monkeypatch):
    src = {"a.cu": "kernel a\n"}
    sha = hashlib.sha256(src["a.cu"].encode()).hexdigest()[:16]
    _write_tree(str(tmp_path), "k", src, "a.cu gone.cu", sha, "1")     # a listed file is missing
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k") is None

