"""The oracle reproduces its stored expected values (regression guard)."""
import os

import numpy as np

import oracle
from tests.golden import make_golden


def load_rows():
    path = os.path.join(os.path.dirname(make_golden.__file__), "small_vanilla_rows.txt")
    rows, lse, out = [], [], []
    for line in open(path):
        if line.startswith("#"):
            continue
        f = line.split()
        rows.append(tuple(int(x) for x in f[:3]))
        lse.append(float(f[3]))
        out.append([float(x) for x in f[4:]])
    return np.array(rows), np.array(lse), np.array(out)


def test_oracle_matches_golden():
    rows, lse, out = load_rows()
    q, k, v = make_golden.small_vanilla_inputs()
    o, l = oracle.attention(q, k, v, rows=rows)
    assert np.max(np.abs(o - out)) < 1e-12
    assert np.max(np.abs(l - lse)) < 1e-12
