"""bench.py's JSON lines, run as the driver runs them (subprocesses, small workload).

The reference arm (the CPU oracle) needs no GPU and runs everywhere; the prefill and
quantise lines need the GB300.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = "prefill_1k_h8kv1_bsm50"
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def _line(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _line("--impl", "reference", "--steps", "1", "--warmup", "1", "--workload", SMALL)
    assert BASE_KEYS <= d.keys()
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == SMALL
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_prefill_line():
    d = _line("--steps", "5", "--warmup", "3", "--workload", SMALL, "--no-cpu-baseline")
    assert BASE_KEYS <= d.keys()
    assert d["value"] > 0 and d["gpu_launches"] == 5
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["host_link"]["h2d_gbs"] > 0 and e["host_link"]["d2h_gbs"] > 0
    assert e["call"].startswith("bsa_fp8_prefill_host")
    assert d["warm_l2_ms_per_call"]["median"] > 0
    assert "sm_mhz" in d["clocks"]
    # the other full-size workloads, timed the same way, in the same line
    import bench

    assert set(d["other_workloads"]) == set(bench.OTHER_WORKLOADS)
    for name, o in d["other_workloads"].items():
        assert o["config"]["workload"] == name and o["value"] > 0
        assert o["roofline"]["frac"] == pytest.approx(o["value"] / o["roofline"]["peak"])


@pytest.mark.gpu
def test_quantise_line():
    d = _line("--op", "quantize", "--steps", "3", "--warmup", "3", "--workload", SMALL)
    assert BASE_KEYS <= d.keys()
    assert d["value"] > 0 and d["roofline"]["bound"] == "hbm"
    assert d["config"]["op"] == "quantize" and d["gpu_launches"] == 6
    pk = d["per_kernel"]
    assert set(pk) == {"quantize_rows_kernel", "append_kv_kernel"}
    assert sum(k["bytes"] for k in pk.values()) == d["config"]["bytes_per_step"]
