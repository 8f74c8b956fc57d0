"""bench.py's host-side contract, no GPU: the traffic figure follows the kernel
sources it was measured on, and the reference arm (the CPU oracle) prints one
JSON line of the required shape."""
import json
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_is_withheld_for_other_sources(tmp_path, monkeypatch):
    prof = tmp_path / "p.md"
    prof.write_text("kernel_source_hash: 0000000000000000\ndram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(prof))
    assert bench.profiled_traffic() is None
    prof.write_text(f"kernel_source_hash: {bench.kernel_source_hash()}\ndram_bytes_per_launch: 123\n")
    assert bench.profiled_traffic() == 123
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.md"))
    assert bench.profiled_traffic() is None


def test_reference_arm_prints_one_line_of_the_contract(monkeypatch, capsys):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    args = types.SimpleNamespace(gpus=1, steps=2, warmup=1, ref_seconds=1.5, workload="softmax_T8192_E2304_k36")
    assert bench.run_reference(args) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["config"]["T"] == 8192 and d["config"]["E"] == 2304 and d["config"]["topk"] == 36
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
