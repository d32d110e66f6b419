"""bench.py on a GPU prints one JSON line with every key of its contract.

A short run of the default workload (few steps, short CPU-baseline sample):
the metric and config, the roofline object (bound, achieved, peak, frac,
traffic), the CPU baseline, the end-to-end leg with host-copy byte counts,
the clock record and the launch count, each with a sane value; the
per-workload entries of every configuration of the suite.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def test_bench_line_has_every_key():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "400", "--warmup", "3",
           "--soak-seconds", "0.6", "--e2e-steps", "4", "--cpu-seconds", "0.3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "cpu_baseline", "e2e", "clocks", "gpu_launches", "nonempty_cta_fraction"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 400 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is False and d["unit"] == "us"
    assert abs(d["ms_per_step"] * 1e3 - d["value"]) < 1e-6 * d["value"] + 1e-9
    assert d["config"]["workload"] == "gqa_ctx5900" and "l2" in d["config"]
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["peak"] > 0 and 0 < roof["frac"] < 2
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert roof["traffic"] is None or roof["traffic"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    pc = d["per_config"]
    for name in ("tiny_gqa_ctx260", "gqa_ctx5900", "fp8_batch8_ctx32k", "mla_t6_ctx64k",
                 "mixed_batch32_bf16", "mixed_batch32_fp8"):
        e = pc[name]
        assert e["us_per_call"] > 0 and e["kernel_us"] > 0 and 0 < e["frac"] < 2, name
        assert e["nonempty_cta_fraction"] == 1.0, name
    assert pc["mla_t6_ctx64k"]["roofline_bound"] == "tensor"
    assert pc["gqa_ctx5900"]["us_per_call"] == d["value"]
    sw = d["split_sweep"]
    assert sw["num_splits"] == [1, 2, 4, 8, 16, 32, 64]
    assert all(f == 1.0 for f in sw["nonempty_cta_fraction"])
    assert sw["kernel_us"][-1] < sw["kernel_us"][0] / 8  # splitting pays
    cp = d["capacity_plan"]
    assert cp["num_splits"] == 64 and cp["planned_items"] == 2 * 64
    assert cp["us_per_call"] > 0 and cp["kernel_us"] > 0 and cp["nonempty_cta_fraction"] == 1.0
    e2e = d["e2e"]
    assert e2e["value"] > d["value"] and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["clocks"]["sm_max_mhz"] > 0 and isinstance(d["clocks"]["reasons"], list)
    assert d["gpu_launches"] == 400 * 2  # split kernel + combine kernel per call
    assert d["nonempty_cta_fraction"] == 1.0
    assert d["cold_us_per_call"] > 0
