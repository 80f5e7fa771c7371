"""bench.py's reference arm (the fp64 oracle on the host cores) runs without a GPU, so its
JSON line, the one the reference arm must print, is checked here key by key."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out
    j = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert j["impl"] == "reference"
    assert j["metric"] == bench.METRIC and j["unit"] == bench.UNIT == "tokens/s"
    assert j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == 3 and j["warmup"] == 3
    assert j["value"] > 0 and j["ms_per_step"] > 0 and j["vs_baseline"] is None
    assert j["data"] == "synthetic" and j["scaling"] == "weak"
    assert j["config"]["workload"] == "chat_wave_32x1024"
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == j["value"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_clock_summary_keeps_the_loaded_window():
    """The clock summary reports only samples taken inside the window the bench sets (its
    timed steps and their untimed tail), with the throttle reasons seen there."""
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, {th}, {pc}"
    c.lines = [(1.0, row.format(sm=1200, th="Not Active", pc="Not Active")),   # before
               (2.0, row.format(sm=2070, th="Not Active", pc="Active")),
               (2.1, row.format(sm=2055, th="Not Active", pc="Not Active")),
               (2.2, row.format(sm=2070, th="Not Active", pc="Not Active")),
               (9.0, row.format(sm=300, th="Active", pc="Not Active"))]          # after
    c.window = (1.5, 3.0)
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    c.window = None
    assert c.summary()["samples"] == 5
    assert "sw_thermal_slowdown" in c.summary()["reasons"]
