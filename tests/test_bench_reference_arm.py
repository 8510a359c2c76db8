"""The benchmark's reference arm on the CPU: the oracle timed on a small
sample of the 7x7 workload, and the JSON line built from such samples, with
the keys the benchmark contract asks for."""
import json
import os
import sys

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))

import bench  # noqa: E402

REQUIRED = ["impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"]


def test_oracle_sample_on_host_cores():
    r = bench.cpu_baseline_conv7x7(target_s=0.05)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s"
    assert r["value"] > 0 and r["seconds"] > 0 and r["cores"] >= 1
    assert "conv7x7_16x64x64x512_to512" in r["sample"]


def test_reference_line_keys():
    samples = [{"value": 0.02, "seconds": 1.5, "cores": 8, "sample": "s"},
               {"value": 0.03, "seconds": 1.0, "cores": 8, "sample": "s"},
               {"value": 0.01, "seconds": 2.0, "cores": 8, "sample": "s"}]
    line = bench.reference_line(samples, gpus=1, steps=3, warmup=3)
    json.dumps(line)
    for k in REQUIRED:
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] == 0.02 and line["ms_per_step"] == 1500.0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["config"]["workload"] == bench.HEADLINE
