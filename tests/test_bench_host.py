"""Host-side measurement arithmetic of bench.py, on CPU: the pairs inside the
visited key tiles (reported beside the unmasked-pair throughput so the work
spent on masked pairs of partial tiles shows) against a brute-force count of
the tiles that hold at least one allowed pair, and the per-step spread."""
from __future__ import annotations

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import testdata  # noqa: E402


def _brute_visited(mask, S, bn, window=0, prefix=0, starts=None):
    """Every (query block, key tile) whose rectangle holds an allowed pair,
    from the masks' per-pair definitions."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    if mask == "none":
        allowed = np.ones((S, S), bool)
    elif mask == "causal":
        allowed = j <= i
    elif mask == "window":
        allowed = (j <= i) & (i - j < window)
    elif mask == "prefix":
        allowed = (j <= i) | (j < prefix)
    else:
        doc = np.searchsorted(np.asarray(starts), np.arange(S), side="right") - 1
        allowed = (doc[:, None] == doc[None, :]) & (j <= i)
    total = 0
    for q0 in range(0, S, 128):
        q1 = min(q0 + 128, S)
        for t0 in range(0, S, bn):
            t1 = min(t0 + bn, S)
            if allowed[q0:q1, t0:t1].any():
                total += (q1 - q0) * (t1 - t0)
    return total


@pytest.mark.parametrize("bn", [64, 112, 128])
@pytest.mark.parametrize("mask,kw", [("none", {}), ("causal", {}), ("window", {"window": 100}),
                                     ("prefix", {"prefix": 170}), ("doc", {})])
@pytest.mark.parametrize("S", [1, 200, 333])
def test_visited_pairs_match_brute_force(S, mask, kw, bn):
    doc = testdata.doc_offsets(S, 2, f"visited{S}", lo=20, hi=150) if mask == "doc" else None
    got = bench.visited_pairs(mask, 2, 3, S, bn, kw.get("window", 0), kw.get("prefix", 0), doc)
    want = sum(_brute_visited(mask, S, bn, kw.get("window", 0), kw.get("prefix", 0),
                              None if doc is None else doc[b]) for b in range(2)) * 3
    assert got == want
    assert got >= bench.unmasked_pairs(mask, 2, 3, S, kw.get("window", 0), kw.get("prefix", 0), doc)


def test_spread():
    s = bench.spread([1.0, 2.0, 3.0, 10.0])
    assert s["median_ms"] == 2.5
    assert abs(s["std_ms"] - float(np.std([1.0, 2.0, 3.0, 10.0]))) < 1e-4
    assert bench.spread([4.0]) == {"median_ms": 4.0, "std_ms": 0.0}
