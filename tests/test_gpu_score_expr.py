"""GPU parity of score_mod expressions (FL_MOD_EXPR) with the expression oracle.

The standard kernel is compiled at run time with each expression as its
score_mod and compared, element by element, with ``oracle.score_expr`` (the
expression evaluated in float64 on the full score matrix, then the plain
softmax) on seeded inputs with ragged last tiles; expressions equivalent to a
built-in variant are also compared with the built-in kernel's output.
"""
from __future__ import annotations

import numpy as np
import pytest

import testdata
from oracle import score_expr as se

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402

CASES = [
    # (expression, mask, B, S, Hq, Hk)
    ("20 * tanh(score / 20)", "none", 2, 333, 4, 4),
    ("score - 0.25 * abs(q_idx - kv_idx)", "causal", 2, 333, 4, 4),
    ("where(kv_idx <= q_idx, score, -inf)", "none", 1, 400, 2, 2),
    ("score * (1 + 0.5 * tanh(h - 1)) + where(b == 1, 0.3, -0.2) * floor(kv_idx / 64)", "none",
     2, 300, 4, 2),
    ("max(score, -2) - exp2(-(h + 1) / 2) * abs(q_idx - kv_idx) / 16", "causal", 1, 520, 8, 2),
    ("where(q_idx < 5, -inf, score)", "none", 1, 200, 2, 2),  # rows 0..4 have no key
]


def _inputs(tag, B, S, Hq, Hk):
    q = testdata.normal_bf16((B, S, Hq, 64), f"expr_{tag}", "q")
    k = testdata.normal_bf16((B, S, Hk, 64), f"expr_{tag}", "k")
    v = testdata.normal_bf16((B, S, Hk, 64), f"expr_{tag}", "v")
    return q, k, v


@pytest.mark.parametrize("expr,mask,B,S,Hq,Hk", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_expression_matches_oracle(expr, mask, B, S, Hq, Hk):
    q, k, v = _inputs(str(testdata.fnv1a64(expr) % 997), B, S, Hq, Hk)
    o, lse, _, err = gu.run_standard(q, k, v, score_expr=expr, mask=mask)
    assert err == 0
    oref, lref = se.attention_expr(q, k, v, expr, mask=mask)
    gu.compare(o, lse, oref, lref, what=f"expr {expr!r} mask={mask}")


def test_expression_equal_to_builtin_variants():
    # the same variant as a built-in score_mod and as an expression: both match
    # the oracle, and each other to the output's bf16 rounding
    B, S, Hq, Hk = 2, 333, 4, 4
    q, k, v = _inputs("builtin", B, S, Hq, Hk)
    pairs = [
        (dict(score_mod="softcap", softcap=20.0), "20 * tanh(score / 20)", "none"),
        (dict(score_mod="none", mask="causal"), "where(kv_idx <= q_idx, score, -inf)", "none"),
        (dict(score_mod="alibi", mask="causal"),
         "score - exp2(-8 * (h + 1) / 4) * abs(q_idx - kv_idx)", "causal"),
    ]
    for builtin, expr, mask in pairs:
        o1, l1, _, e1 = gu.run_standard(q, k, v, **builtin)
        o2, l2, _, e2 = gu.run_standard(q, k, v, score_expr=expr, mask=mask)
        assert e1 == 0 and e2 == 0
        oref, lref = se.attention_expr(q, k, v, expr, mask=mask)
        gu.compare(o2, l2, oref, lref, what=f"expr {expr!r}")
        assert np.abs(o1 - o2).max() <= 2 ** -7, f"{expr!r}: built-in and expression differ"
        assert np.abs(l1 - l2).max() <= 1e-3


def test_expression_with_sequence_mask_on_top():
    # the desc's window mask still applies after the expression
    B, S, Hq, Hk = 1, 300, 2, 2
    q, k, v = _inputs("window", B, S, Hq, Hk)
    expr = "score + 0.1 * h"
    o, lse, counts, err = gu.run_standard(q, k, v, score_expr=expr, mask="window", window=64)
    assert err == 0
    # window 64 = causal plus "q_idx - kv_idx < 64" written into the expression
    oref, lref = se.attention_expr(q, k, v, "where(q_idx - kv_idx < 64, score + 0.1 * h, -inf)",
                                   mask="causal")
    gu.compare(o, lse, oref, lref, what="expr + window mask")


def test_bad_expression_launches_nothing():
    import attention_variant_gb300 as fa

    q, k, v = _inputs("bad", 1, 128, 2, 2)
    with pytest.raises(fa.FlAttnError) as ei:
        gu.run_standard(q, k, v, score_expr="score ** 2")
    assert ei.value.status == fa.FL_ERR_INVALID_ARG
