"""bench.py's JSON line on the GPU: one line with every key of the
benchmark contract, on the tiny workload (the per-workload breakdown and the
CPU baseline still run, so this takes about a minute)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keeps_the_contract():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny", "--steps", "5",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    out = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in out, key
    assert out["value"] > 0 and out["n_gpus"] == 1 and out["steps"] == 5 and out["warmup"] >= 3
    assert out["higher_is_better"] is True and out["scaling"] == "weak" and out["dtype"] == "fp32"
    assert out["vs_baseline"] is None and "workload" in out["config"]
    roof = out["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    cpu = out["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]
    e2e = out["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert out["gpu_launches"] == 2 * 5  # forward and backward per step, one launch each
    clocks = out["clocks"]
    assert clocks["sm_max_mhz"] > 0 and isinstance(clocks["reasons"], list)
    # several timed regions of K steps; value and ms_per_step from the median
    reg = out["timed_regions"]
    assert reg["count"] >= 5 and reg["steps_each"] == 5
    assert reg["min_ms"] <= reg["median_ms"] <= reg["max_ms"]
    assert abs(out["ms_per_step"] - reg["median_ms"] / 5) < 1e-3
    # the token split at one rank is the named workload, one run
    assert out["config"]["split"]["mode"] == "tokens" and out["plan"]["runs_per_direction"] == 1
    assert 0 < roof["frac_of_nominal"] < roof["frac"]
    # per-workload entries name their figure of record; notes explain the labels
    wl = out["workloads"]
    assert wl["gqa"]["fwd"]["of_record"] == "steady_frac" and "notes" in wl
    assert wl["small_model"]["fwd"]["graph_l2_resident"] is True
    assert wl["e2e_gqa"]["value"] > 0 and wl["e2e_gqa"]["host_link"]["both_GB/s"] > 0
