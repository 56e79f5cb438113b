"""GPU probe of the design's hardware numbers (tests/probes/hw_probe.cu): the
exponential unit's rate and the tcgen05 MMA shapes the forward kernel issues.
The figures are printed (run with -s to see them) and checked against wide
plausibility bounds only; the design text quotes the measured values."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "tiled_online_softmax_fwd_gb300", "csrc")


def run_probe(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = os.path.join(tmp_path, "hw_probe")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", CSRC, "-o", exe, os.path.join(HERE, "probes", "hw_probe.cu")],
                   check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    figures = {}
    for line in out.splitlines():
        assert not line.startswith("error"), line
        parts = line.split()
        if parts[0] == "sms":
            figures["sms"] = int(parts[1])
        elif parts[0].startswith("mufu"):
            figures[parts[0]] = float(parts[1])
        elif parts[0].startswith("mma_"):
            figures[parts[0]] = (float(parts[2]), float(parts[4]))
    return out, figures


def test_hw_probe(tmp_path):
    out, f = run_probe(tmp_path)
    print(out)
    assert f["sms"] > 0
    # Exponentials per clock per SM: a power of two between 8 and 128 on any
    # recent part (16 lanes per SMSP quarter-rate would be 16).
    assert 8.0 <= f["mufu_ex2_per_clk_per_sm"] <= 160.0
    # The dense shapes reach at least half of 8192 FLOP/clk/SM.
    for key in ("mma_s_ss_128x128x16", "mma_pv_ts_128x128x16", "mma_s_ss_128x256x16"):
        assert f[key][1] >= 4096.0, key
    # Every shape finishes (no timed-out wait) with a positive rate.
    for key, v in f.items():
        if key.startswith("mma_"):
            assert v[0] > 0 and v[1] > 0, key
