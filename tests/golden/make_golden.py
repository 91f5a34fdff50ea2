"""Writes tests/golden/cfg0_oracle_sample.txt from the fp64 oracle alone.

The pages print no numeric example of the gated delta rule, so this file is a
regression fixture, not a page value: it freezes a sample of the oracle's
outputs on the tiny config (1 sequence, T=128, 2 heads, d=64, seed 0) so that
an unintended change to the oracle's arithmetic shows up as a diff. It calls
only `oracle` and the seeded input generators.

Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cfg0_oracle_sample.txt")

# (token, head, column) of the outputs and (head, row, column) of the final state
O_IDX = [(0, 0, 0), (0, 1, 63), (1, 0, 5), (17, 1, 30), (63, 0, 62), (64, 1, 1), (65, 0, 40),
         (100, 1, 7), (127, 0, 0), (127, 1, 63)]
S_IDX = [(0, 0, 0), (0, 63, 63), (1, 10, 20), (1, 63, 0), (0, 31, 32)]


def sample():
    w = workloads.config(0)
    o, s = oracle.run_workload(w)
    return ([(i, float(o[i])) for i in O_IDX], [(i, float(s[(0,) + i])) for i in S_IDX],
            float(np.sqrt((o ** 2).sum())), float(np.sqrt((s ** 2).sum())))


def main():
    os_, ss, on, sn = sample()
    with open(OUT, "w") as f:
        f.write("# fp64 oracle on config 0 (seed 0); written by make_golden.py\n")
        f.write("# kind index value\n")
        for i, v in os_:
            f.write(f"o {i[0]} {i[1]} {i[2]} {v!r}\n")
        for i, v in ss:
            f.write(f"s {i[0]} {i[1]} {i[2]} {v!r}\n")
        f.write(f"o_fro {on!r}\ns_fro {sn!r}\n")


if __name__ == "__main__":
    main()
