"""Host logic of bench.py that needs no GPU: the reference arm's JSON line
(the CPU oracle on a small table) and the rule that committed ncu traffic
figures are reported only for the workload and the decoder sources they were
captured on."""

import contextlib
import io
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--rows", "20000", "--steps", "2", "--warmup", "3"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_reference_arm_rejects_short_warmup():
    try:
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "2"])
    except SystemExit as e:
        assert "warmup" in str(e)
    else:
        raise AssertionError("a warm-up below 3 steps must be refused")


def test_traffic_record_matches_sources():
    rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    for f in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(ROOT, "host_transfer_gb300", "csrc", f)), f
    for config, legs in rec.items():
        for kind, ent in legs.items():
            assert os.path.exists(os.path.join(ROOT, ent["source"])), ent["source"]
            assert ent["dram_bytes_read"] >= 0 and ent["dram_bytes_write"] >= 0
            assert len(ent["kernel_source_sha256"]) == 64


def test_traffic_only_for_current_sources_and_workload(monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    ent = rec["dense_gnn"]["hbm_resident"]
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: ent["kernel_source_sha256"])
    got = bench.kernel_traffic("hbm_resident", "dense_gnn")
    assert got["dram"] == ent["dram_bytes_read"] + ent["dram_bytes_write"]
    assert bench.kernel_traffic("hbm_resident", "no_such_workload") == {}
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "0" * 64)
    assert bench.kernel_traffic("hbm_resident", "dense_gnn") == {}
