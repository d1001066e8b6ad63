"""bench.py --impl reference on CPU: the oracle timed on the host, one JSON line in the contract's
shape (the same metric, unit and direction as the GPU arm, a cpu_baseline and an e2e object with no
host-device bytes)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    import bench
    assert r["impl"] == "reference" and r["metric"] == bench.METRIC
    assert r["unit"] == "tokens/s" and r["higher_is_better"] is True and r["scaling"] == "weak"
    assert r["steps"] == 2 and r["warmup"] == 1 and r["n_gpus"] == 1
    assert r["value"] > 0 and r["ms_per_step"] > 0 and r["vs_baseline"] is None
    assert r["config"]["workload"].startswith("tiny") and r["config"]["T"] == 256
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == r["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = r["e2e"]
    assert e2e["value"] == r["value"] and e2e["unit"] == r["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
