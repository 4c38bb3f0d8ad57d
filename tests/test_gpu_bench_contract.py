"""bench.py's JSON line keeps its contract: one line on stdout with the
metric, the whole-job value, the timing fields, the roofline of the dominant
kernel, the oracle's CPU baseline, the end-to-end figure with its copy bytes,
the launch count and the clock record.  Run on the 32k workload (a small
case: about a minute on one GPU)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_every_contract_key():
    cmd = [sys.executable, "bench.py", "--workload", "bf16_32k", "--steps", "2", "--warmup", "3", "--e2e-steps", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key, typ in (("metric", str), ("value", (int, float)), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", (int, float)), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("roofline", dict), ("cpu_baseline", dict),
                     ("e2e", dict), ("gpu_launches", int), ("clocks", dict)):
        assert isinstance(d.get(key), typ), (key, d.get(key))
    assert "vs_baseline" in d
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "bf16_32k"
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor", "l2", "alu")
    for key in ("achieved", "peak", "frac", "unit"):
        assert key in rf, key
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-2)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    ck = d["clocks"]
    assert "sm_mhz" in ck and "sm_max_mhz" in ck and "reasons" in ck
