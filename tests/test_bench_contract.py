"""The bench's output contract, checked on the CPU through its reference arm
(the oracle timed on the host cores): one JSON line carrying the keys a reader
of the line relies on, with the warm-up floor applied and the value derived
from the counted flops of one (b, h) head per step."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "impl", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2
    assert d["warmup"] >= 3   # at least three warm-up steps, whatever is asked for
    assert d["higher_is_better"] is True and d["vs_baseline"] is None and d["unit"] == "TFLOP/s"
    assert d["config"]["workload"] == "keypad_fp16_b8h8s2048d64"
    # fwd (4 D) + bwd (10 D) flops per (q, kv) pair of one 2048 x 2048 head, over the mean step time
    want = 14.0 * 2048 * 2048 * 64 / (d["ms_per_step"] * 1e-3) / 1e12
    assert d["value"] > 0 and abs(d["value"] - want) <= 1e-9 * want
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["host_cpus"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
