"""bench.py --impl reference (CPU only): the oracle timed on the host cores
prints one JSON line with the same metric, unit and direction as the GPU arm,
marked as the reference, with an end-to-end figure that moves no bytes and a
cpu_baseline describing the sample.  Run on the small workload so the suite
stays fast; the metric string names the workload it was measured on."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
         "--warmup", "1", "--workload", "tiny_b1h2s256d64_f16"],
        cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    # at least three warm-up steps are always run (and reported), whatever was asked
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"]
    assert d["config"]["workload"] == "tiny_b1h2s256d64_f16"
    assert "no GPU L2" in d["config"]["l2"]
