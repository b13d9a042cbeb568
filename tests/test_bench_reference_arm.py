"""The benchmark's reference arm (`bench.py --impl reference`) on the CPU: it
times the fp64 oracle and prints the benchmark's one-line JSON record, with
the keys every bench line carries and those of a reference line (impl,
cpu_baseline, an end-to-end figure with no host-device copies)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
         "--steps", "2", "--warmup", "0"],
        capture_output=True, text=True, timeout=600, cwd=ROOT, check=True).stdout
    lines = [x for x in out.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "unit", "n_gpus", "ms_per_step", "scaling", "dtype", "data"):
        assert key in d, key
    assert d["steps"] == 2 and d["warmup"] == 3  # at least three warm-up steps
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "rows" in cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
