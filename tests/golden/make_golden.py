"""Write tests/golden/oracle_B1_H1_N256_d64.txt.

Calls only the fp64 oracle (oracle/) and the seeded input generator.  The file
freezes the oracle's output on the smallest workload (B=1, H=1, N=256, d=64,
non-causal, seed 0, scale 1/sqrt(64)), so that any later change to the oracle's
arithmetic or to the input recipe shows up as a failing CPU test.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from tiled_online_softmax_fwd_gb300.inputs import WORKLOADS, digest, make_workload  # noqa: E402

ROWS_WITH_O = [0, 1, 127, 128, 255]


def main():
    w = WORKLOADS["B1_H1_N256_d64"]
    q, k, v, _ = make_workload(w)
    o, lse = oracle.attn_fwd(q, k, v, w.scale, w.causal)
    path = os.path.join(HERE, "oracle_B1_H1_N256_d64.txt")
    with open(path, "w") as f:
        f.write("# fp64 oracle output, written by tests/golden/make_golden.py\n")
        f.write("# workload B=1 H=1 N=256 d=64 non-causal seed=0 scale=%r\n" % w.scale)
        f.write("digest %s\n" % digest(q, k, v))
        for i in range(w.N):
            f.write("lse %d %.17g\n" % (i, lse[i]))
        for i in ROWS_WITH_O:
            f.write("o %d %s\n" % (i, " ".join("%.17g" % x for x in o[i])))
    print("wrote", path)


if __name__ == "__main__":
    main()
