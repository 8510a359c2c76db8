"""Host logic of the benchmark (no GPU): the DRAM-traffic figure is reported
only while the kernel sources it was captured from are unchanged, and the
roofline object carries the fields the benchmark line promises."""
import json
import os
import sys

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))

import bench  # noqa: E402


def _tree(tmp_path, source_text):
    csrc = tmp_path / "gemm_conv_epilogues_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(source_text)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_traffic_only_while_sources_unchanged(tmp_path, monkeypatch):
    csrc = _tree(tmp_path, "// kernel source\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entry = {"files": ["k.cu"], "files_sha256_16": bench.files_fingerprint(["k.cu"]),
             "dram_bytes_per_launch": 123456789}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"w": entry}))
    assert bench.kernel_traffic("w") == 123456789.0
    assert bench.kernel_traffic("other") is None
    (csrc / "k.cu").write_text("// kernel source, edited\n")
    assert bench.kernel_traffic("w") is None


def test_traffic_absent_file(tmp_path, monkeypatch):
    _tree(tmp_path, "x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("w") is None


def test_committed_traffic_entries_name_existing_sources():
    t = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert set(t) >= {"conv7x7_16x64x64x512_to512", "conv1x1_32x56x56x256_to256", "bias_gelu_f16_8192x8192",
                      "bias_gelu_rowsum_f16_8192x8192", "residual_layernorm_f16_16384x4096"}
    for w, e in t.items():
        for f in e["files"]:
            assert os.path.exists(os.path.join(bench.ROOT, "gemm_conv_epilogues_gb300", "csrc", f)), (w, f)
        assert e["dram_bytes_per_launch"] == e["dram_read"] + e["dram_write"] or \
            abs(e["dram_bytes_per_launch"] - e["dram_read"] - e["dram_write"]) <= 2


def test_roofline_fields():
    r = bench.roofline("tensor", 1900.0, 1943.5, "TFLOP/s", 1.6e8)
    assert r == {"bound": "tensor", "achieved": 1900.0, "peak": 1943.5, "unit": "TFLOP/s",
                 "frac": round(1900.0 / 1943.5, 4), "traffic": 1.6e8}
