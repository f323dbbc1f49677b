"""The reference arm of bench.py (the CPU oracle on the host's cores, here two processes) keeps the JSON-line
contract: one line with impl "reference", the window metric in us/window (lower is better), a
cpu_baseline naming the cores it used, and an e2e object with no host<->device bytes."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--ref-procs", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == "us_per_verify_window_48L" and d["unit"] == "us/window"
    assert d["higher_is_better"] is False and d["steps"] == 1 and d["warmup"] >= 3
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    assert d["cpu_baseline"]["cores"] == min(2, cores) and d["cpu_baseline"]["kind"] == "oracle"
    assert d["config"]["parallelism"] == f"{min(2, cores)} CPU processes"
    assert d["e2e"] == {"value": d["value"], "unit": "us/window", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
