"""CPU test: the oracle and the input recipe still reproduce the frozen golden
file (written by tests/golden/make_golden.py, which calls only the oracle)."""
import os

import numpy as np

import oracle
from tiled_online_softmax_fwd_gb300.inputs import WORKLOADS, digest, make_workload

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "oracle_B1_H1_N256_d64.txt")


def _read():
    lse, o, dig = {}, {}, None
    for line in open(GOLDEN):
        if line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] == "digest":
            dig = parts[1]
        elif parts[0] == "lse":
            lse[int(parts[1])] = float(parts[2])
        elif parts[0] == "o":
            o[int(parts[1])] = np.array([float(x) for x in parts[2:]])
    return dig, lse, o


def test_golden_oracle_output():
    dig, lse_g, o_g = _read()
    w = WORKLOADS["B1_H1_N256_d64"]
    q, k, v, _ = make_workload(w)
    assert digest(q, k, v) == dig, "input recipe changed"
    o, lse = oracle.attn_fwd(q, k, v, w.scale, w.causal)
    for i, x in lse_g.items():
        assert abs(lse[i] - x) <= 1e-13 * max(1.0, abs(x))
    for i, row in o_g.items():
        assert np.max(np.abs(o[i] - row)) <= 1e-13
