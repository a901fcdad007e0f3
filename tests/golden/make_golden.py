"""Write the stored expected values under tests/golden/ (calls only the oracle).

Run from the repository root:  python tests/golden/make_golden.py

small_vanilla_rows.txt: the small vanilla MHA problem (B=1, H=2, S=256, D=64,
scale 1/8, inputs N(0,1) bf16 from the shared seeded generator) at sampled
rows.  Each line is ``b h i lse o_0 ... o_63`` in float64 (repr).
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import testdata  # noqa: E402
from testdata import workloads  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
ROWS = [(0, h, i) for h in (0, 1) for i in (0, 1, 63, 127, 128, 200, 255)]


def small_vanilla_inputs():
    w = workloads.SMALL_VANILLA
    shape = (w["B"], w["S"], w["H"], w["D"])
    return tuple(testdata.normal_bf16(shape, w["name"], t) for t in ("q", "k", "v"))


def main():
    q, k, v = small_vanilla_inputs()
    o, lse = oracle.attention(q, k, v, rows=np.array(ROWS))
    path = os.path.join(HERE, "small_vanilla_rows.txt")
    with open(path, "w") as f:
        f.write("# b h i lse o[0..63]; oracle output for the small vanilla MHA problem\n")
        for n, (b, h, i) in enumerate(ROWS):
            vals = " ".join(repr(float(x)) for x in o[n])
            f.write(f"{b} {h} {i} {float(lse[n])!r} {vals}\n")
    print(path)


if __name__ == "__main__":
    main()
