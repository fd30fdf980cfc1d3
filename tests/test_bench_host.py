"""bench.py's host-side arms, no GPU: the reference arm (the oracle on a sampled
decode step) prints one well-formed JSON line, and the all-cores oracle pool
runs a step."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_all_cores_oracle_pool():
    sys.path.insert(0, ROOT)
    import bench
    res = bench.cpu_baseline_all_cores(1)
    assert res["value"] > 0 and res["cores"] == (os.cpu_count() or 1)
