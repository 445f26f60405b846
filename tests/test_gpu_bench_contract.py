"""bench.py's own arm keeps the JSON-line contract on a GPU: one line with the
metric, value, step counts, roofline (with the measured peak), clocks sampled
during the timed region, gpu_launches, the e2e object fed through the C ABI
from host memory, and the CPU-oracle baseline.  Run on the small GPT-2-shaped
set so it takes seconds."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, p.stdout[-2000:]
    return json.loads(lines[0])


def test_step_bench_json_line():
    d = _bench("--workload", "gpt2_small", "--steps", "4", "--warmup", "3",
               "--cpu-seconds", "2")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "clocks", "gpu_launches", "e2e", "cpu_baseline"):
        assert k in d, k
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "params/s" and d["scaling"] == "weak"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    c = d["clocks"]
    assert c["sm_mhz"] > 0 and isinstance(c["reasons"], list)
    assert d["gpu_launches"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # copies run back to back inside the timed region: their busy time per
    # step cannot exceed the step
    assert e["h2d_copy_ms"]["mean_busy"] <= e["ms_per_step"] * (1 + 1e-6)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert cb["host_nproc"] >= 1 and cb["cpu_model"]


def test_sweep_bench_json_line():
    for gran in ("tensorwise", "groupwise"):
        d = _bench("--workload", "fp8_sweep", "--fp8-granularity", gran, "--steps", "3",
                   "--warmup", "3", "--no-e2e", "--no-cpu-baseline")
        assert d["unit"] == "GB/s" and d["value"] > 0 and d["roofline"]["peak"] > 0
        assert d["gpu_launches"] > 0
