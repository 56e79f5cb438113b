"""GPU smoke tests of bench.py's own legs: each prints one parseable JSON line
with the keys the contract asks for."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_small_workload_line():
    j = bench("--workload", "B1_H1_N256_d64", "--steps", "5", "--warmup", "3",
              "--cpu-budget", "0.5")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in j, key
    assert j["value"] > 0 and j["step_quantiles_ms"]["p50"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] > 0


def test_decode_line():
    j = bench("--op", "decode_B2_H32_Nq1_Nk32768_d128", "--steps", "5", "--warmup", "3",
              "--cpu-budget", "0.5")
    assert j["unit"] == "GB/s" and j["value"] > 0 and j["roofline"]["bound"] == "hbm"
    assert j["e2e"]["h2d_bytes_per_step"] > 0


def test_reference_line():
    j = bench("--impl", "reference", "--steps", "2", "--warmup", "1")
    assert j["impl"] == "reference" and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0
