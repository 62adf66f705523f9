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


def _reference_line(argv):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", *argv])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def _check_reference(d, steps, warmup):
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == steps and d["warmup"] == warmup and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_line():
    d = _reference_line(["--config", "dense_gnn", "--rows", "20000", "--steps", "2", "--warmup", "3"])
    _check_reference(d, 2, 3)
    args = bench.parse_args(["--config", "dense_gnn", "--rows", "20000"])
    assert d["config"] == bench.config_of("dense_gnn", args, 1)  # the GPU arm prints the same object
    assert "65,536 ids" in d["cpu_baseline"]["sample"]  # a whole batch per step, as on the GPU


def test_reference_arm_llm_decodes_whole_layers():
    """The default config's reference arm: the headline (LLM offload) with
    whole layers per step, as the GPU arm decodes them."""
    d = _reference_line(["--layers", "2", "--steps", "1", "--warmup", "3"])
    _check_reference(d, 1, 3)
    args = bench.parse_args(["--layers", "2"])
    assert d["config"] == bench.config_of("llm", args, 1)
    assert "whole layer" in d["cpu_baseline"]["sample"]


def test_output_ring_exceeds_l2():
    class C:
        l2 = 126 * 2**20

    for out_bytes in (33_554_432, 67_108_864, 100_663_296, 300_000_000):
        n = bench.Ctx.ring_count(C(), out_bytes)
        assert n >= 2 and n * out_bytes >= 2 * C.l2


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
