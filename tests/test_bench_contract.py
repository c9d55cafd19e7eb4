"""The benchmark's reference arm on CPU: the JSON line keeps the contract's keys
(the oracle timed on this host's cores, one bounded sample of the headline
workload's step: every sequence, 4 of its layer decodes)."""
import json
import sys

from conftest import ROOT


def test_reference_arm_line_has_the_contract_keys():
    sys.path.insert(0, ROOT)
    import bench
    line = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), 0, 1)
    json.dumps(line)  # serialisable as one JSON line
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert k in line, k
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["gpu_launches"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert "workload" in line["config"]
