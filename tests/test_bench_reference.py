"""bench.py's reference arm (the CPU oracle) keeps the JSON-line contract:
one line with the metric, the value and its unit, the step counts, the
cpu_baseline and e2e objects, and impl = "reference".  It runs on host cores
only, so it is checked here on the small GPT-2-shaped set."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=600, cwd=ROOT)


def test_reference_arm_json_line():
    p = _run("--impl", "reference", "--workload", "gpt2_small", "--steps", "2", "--warmup", "3")
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in d, k
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "params/s" and d["higher_is_better"] is True
    assert d["config"]["grad_dtype"] == "bf16"
    assert "bf16 grads" in d["storage"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert cb["host_nproc"] >= 1 and cb["cpu_model"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_bench_rejects_short_warmup():
    p = _run("--impl", "reference", "--workload", "gpt2_small", "--steps", "1", "--warmup", "1")
    assert p.returncode != 0
    assert "warmup" in p.stderr
