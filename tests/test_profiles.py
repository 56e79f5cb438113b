"""The committed ncu summaries (profiles/) carry `bench-key` blocks, which
bench.py reads for the roofline's measured DRAM traffic.  Each block names a
known workload, the 16-hex-digit kernel source hash its counters were taken
at, and positive byte counts; bench's lookup finds every block under its own
hash (and only there: a summary of another source gives no traffic)."""
import glob
import os
import re

import pytest

import bench
from tiled_online_softmax_fwd_gb300.inputs import KV_WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _blocks():
    out = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        cur = None
        for line in open(path):
            if not line.startswith("bench-key "):
                continue
            k, _, v = line[len("bench-key "):].strip().partition("=")
            if k == "workload":
                cur = {"_file": os.path.basename(path)}
                out.append(cur)
            assert cur is not None, "%s: a bench-key before any workload key" % path
            cur[k] = v
    return out


BLOCKS = _blocks()


def test_profiles_carry_bench_keys():
    names = {b["workload"] for b in BLOCKS}
    for w in ("B1_H32_N16384_d128_causal_sigma3", "B2_H8_N65536_d64", "B4_H16_N4096_d128_causal"):
        assert w in names, w
    pairs = [(b["workload"], b["kernel_source"]) for b in BLOCKS]
    assert len(pairs) == len(set(pairs)), "one block per workload and kernel source"


@pytest.mark.parametrize("block", BLOCKS, ids=[b["workload"] for b in BLOCKS])
def test_bench_key_block_is_well_formed(block, monkeypatch):
    assert block["workload"] in set(bench.ALL_WORKLOADS) | set(KV_WORKLOADS)
    assert re.fullmatch(r"[0-9a-f]{16}", block["kernel_source"])
    byte_keys = [k for k in block if k.endswith("bytes_per_launch")]
    assert "dram_bytes_per_launch" in byte_keys
    for k in byte_keys:
        assert int(block[k]) > 0, k
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: block["kernel_source"])
    for k in byte_keys:
        assert bench.profiled_traffic(block["workload"], k) == (int(block[k]), block["_file"])
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic(block["workload"]) == (None, None)
