"""The JSON line bench.py prints: every key the measurement contract names.

The reference arm (the CPU oracle) runs here; the GPU arm is marked gpu. Both
run the small tiny_p4_e16_h256 workload in a subprocess, as a user would.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, steps, warmup):
    assert d["metric"] and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    assert d["dtype"] and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny_p4_e16_h256"
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in d["e2e"], k


def test_reference_arm_line():
    d = _bench("--impl", "reference", "--workload", "tiny_p4_e16_h256", "--steps", "2", "--warmup", "3")
    _common(d, 2, 3)
    assert d["impl"] == "reference"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    # the config is what was timed: here the whole tiny workload fits the budget
    assert d["config"]["sample"] == "full workload" and d["config"]["S"] == 256
    assert "T=64 tokens per rank (S=256" in cb["sample"]


def test_reference_arm_states_a_reduced_sample():
    """With --ref-tokens below the workload's own T, the config names the
    tokens per rank that were timed."""
    d = _bench("--impl", "reference", "--workload", "tiny_p4_e16_h256", "--steps", "2", "--warmup", "3",
               "--ref-tokens", "16")
    assert d["config"]["S"] == 4 * 16 and d["config"]["sample"].startswith("T=16 of the workload's 64")


@pytest.mark.gpu
def test_gpu_arm_line():
    d = _bench("--workload", "tiny_p4_e16_h256", "--steps", "20", "--warmup", "3", "--cpu-seconds", "0.5")
    _common(d, 20, 3)
    assert "impl" not in d or d["impl"] != "reference"
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["achieved"] > 0 and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert "traffic" in rf
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["value"] != d["value"]
    hl = e2e["host_link"]  # the step's copies alone, the ceiling e2e is judged against
    assert hl["h2d_gbs"] > 0 and hl["d2h_gbs"] > 0 and hl["concurrent_gbs"] > 0
    assert hl["e2e_frac_of_concurrent"] == pytest.approx(hl["e2e_gbs"] / hl["concurrent_gbs"])
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert d["gpu_launches"] == 5 * 20
    st = d["stages"]
    assert st["layout_notify_us"] >= 0 and st["layout_notify_event_us"] > 0 and st["layout_notify_method"]
    assert "l2" in d["config"]
