"""The reference arm of bench.py (the oracle timed on the host cores) keeps the
one-JSON-line contract: same metric and workload config as the GPU arm, an
``impl`` tag, a ``cpu_baseline`` describing the run and an ``e2e`` object with no
host-device traffic.  Runs on CPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                        "--config", "tiny"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["metric"] == "spec steps/s" and j["unit"] == "steps/s" and j["higher_is_better"] is True
    assert j["value"] > 0 and j["steps"] == 1 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["config"]["workload"] == "tiny"
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == j["value"]
    e = j["e2e"]
    assert e["value"] == j["value"] and e["unit"] == j["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
