"""Host logic of bench.py that needs no GPU: the reference arm's JSON line
(the CPU oracle timed on this host) and the rule that a committed DRAM-traffic
figure is reported only while its kernel source is unchanged."""
import hashlib
import json
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_complete_json_line(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "0")
    args = types.SimpleNamespace(config=0, steps=1, warmup=0, gpus=1)
    res = bench.run_reference(args)
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1 and json.loads(lines[0]) == res
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in res, key
    assert res["impl"] == "reference" and res["value"] > 0 and res["unit"] == "GB/s"
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["cores"] >= 1
    assert res["e2e"] == {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert res["config"]["workload"] == "m1_k256_n256_int4_bs32_sym_f32"


def test_traffic_is_reported_only_while_the_kernel_source_is_unchanged(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cuh"
    src.write_text("// kernel v1\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"k:w": {"bytes_per_launch": 123.0, "source": "kernel.cuh", "source_sha256_16": h}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k:w") == 123.0
    assert bench.traffic_for("other:w") is None
    src.write_text("// kernel v2\n")
    assert bench.traffic_for("k:w") is None


def test_committed_traffic_entries_name_existing_sources_and_summaries():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    assert table
    for key, e in table.items():
        assert os.path.exists(os.path.join(ROOT, e["source"])), key
        assert os.path.exists(os.path.join(ROOT, e["summary"])), key
        assert e["bytes_per_launch"] == e["dram_read"] + e["dram_write"], key
