"""The driver's JSON line from bench.py on a small table: one line, with the
keys and types the bench contract asks for (roofline, cpu_baseline, e2e,
clocks, gpu_launches) and a bit-exact parity flag."""

import contextlib
import io
import json

import pytest

import bench

pytestmark = pytest.mark.gpu


def _line(argv):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(argv)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_driver_line_keys_on_a_small_table():
    d = _line(["--config", "dense_gnn", "--rows", "40000", "--steps", "3", "--warmup", "3",
               "--cpu-seconds", "0.5"])
    for k, t in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                 ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                 ("dtype", str), ("data", str), ("config", dict), ("gpu_launches", int)):
        assert isinstance(d[k], t), k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert "workload" in d["config"]
    assert d["hbm_resident"]["roofline"]["bound"] == "hbm"
    r = d["roofline"]
    assert r["bound"] == "host_link"  # the headline leg reads the slots over the host link
    assert r["unit"] == "GB/s" and r["peak"] > 0 and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    assert cb["single_thread"]["cores"] == 1 and cb["compress"]["value"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "GB/s" and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= d["steps"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["parity"] == "bit-exact"
