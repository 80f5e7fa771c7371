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
