"""Plant plausible mistakes in a copy of the oracle and check a pin fails.

Each mutant edits one expression of ``oracle/fl_oracle.c`` in a temporary
copy (the committed oracle is never changed), builds it, and runs every pin
of ``tests/oracle_pins.py`` against it.  A mutant that passes every pin would
mean the pins cannot tell that mistake from the definition.
"""
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "fl_oracle.c")

MUTANTS = {
    "causal_strict": ("return j <= i;", "return j < i;"),
    "window_off_by_one": ("i - j < p->window", "i - j <= p->window"),
    "prefix_inclusive": ("j <= i || j < p->prefix", "j <= i || j <= p->prefix"),
    "doc_start_exclusive": ("if (starts[t] <= x)", "if (starts[t] < x)"),
    "doc_no_causal": ("return j <= i && doc_of", "return doc_of"),
    "alibi_sign": ("x += -alibi_slope(p, h)", "x += alibi_slope(p, h)"),
    "alibi_no_abs": ("fabs((double)(i - j))", "((double)(i - j))"),
    "alibi_slope_index": ("-8.0 * (double)(h + 1)", "-8.0 * (double)(h)"),
    "softcap_dropped_cap": ("x = p->softcap * tanh(x / p->softcap);", "x = tanh(x);"),
    "gqa_modulo": ("const int32_t hk = h / group;", "const int32_t hk = h % p->Hk;"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "no_max_subtraction": ("l += exp(z[j] - m);", "l += exp(z[j]);"),
    "scale_one_over_d": ("1.0 / sqrt((double)p->D)", "1.0 / (double)p->D"),
    "bias_transposed": ("i * p->bias_stride[1] +\n                                    j * p->bias_stride[2]",
                        "j * p->bias_stride[1] +\n                                    i * p->bias_stride[2]"),
    "bias_dropped": ("x += widen_bf16(p->bias[", "x += 0.0 * widen_bf16(p->bias["),
    "k_row_uses_q_stride": ("j * p->k_stride[1]", "j * p->q_stride[1]"),
    "v_wrong_row": ("j * p->v_stride[1] + hk", "(p->Sk - 1 - j) * p->v_stride[1] + hk"),
    "softmax_not_normalised": ("const double pj = exp(z[j] - m) / l;", "const double pj = exp(z[j] - m);"),
    "kv_len_inclusive": ("return j < p->kv_len[b];", "return j <= p->kv_len[b];"),
    "decode_position_off_by_one": ("j <= (int64_t)p->kv_len[b] - p->Sq + i", "j < (int64_t)p->kv_len[b] - p->Sq + i"),
    "decode_rows_from_start": ("j <= (int64_t)p->kv_len[b] - p->Sq + i", "j <= i"),
    "key_mask_inverted": ("if (p->key_mask && !p->key_mask[", "if (p->key_mask && p->key_mask["),
    "key_mask_axes_swapped": ("b * p->key_mask_stride[0] + j * p->key_mask_stride[1]",
                              "j * p->key_mask_stride[0] + b * p->key_mask_stride[1]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(text.replace(old, new))
    lib_path = oracle.build(force=True, source=str(mutated), target=str(tmp_path / "libm.so"))
    lib = oracle.load(lib_path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin detects mutant {name}"


# Mistakes planted in the score_mod-expression oracle (oracle/score_expr.py):
# each replaces one entry of its operator or function tables for the duration
# of the test; the expression pin must fail.
def _expr_mutants():
    import ast

    import numpy as np

    return {
        "expr_tanh_is_sinh": ("_FUNCS", "tanh", (1, np.sinh)),
        "expr_le_is_lt": ("_CMP", ast.LtE, np.less),
        "expr_gt_is_ge": ("_CMP", ast.Gt, np.greater_equal),
        "expr_sub_reversed": ("_BIN", ast.Sub, lambda a, b: b - a),
        "expr_div_is_mul": ("_BIN", ast.Div, np.multiply),
        "expr_exp2_is_exp": ("_FUNCS", "exp2", (1, np.exp)),
        "expr_where_swapped": ("_FUNCS", "where", (3, lambda c, x, y: np.where(np.asarray(c) != 0, y, x))),
    }


@pytest.mark.parametrize("name", sorted(_expr_mutants()))
def test_expr_mutant_is_caught(name, monkeypatch):
    from oracle import score_expr as se

    table, key, value = _expr_mutants()[name]
    monkeypatch.setitem(getattr(se, table), key, value)
    with pytest.raises(AssertionError):
        oracle_pins.pin_score_expr(oracle.load())


# Mistakes planted in the backward oracle (oracle.attention_bwd): its source
# is edited in memory, compiled, and swapped in for the duration of the test.
BWD_MUTANTS = {
    "bwd_no_D_term": ("P * (dP - (P * dP).sum(axis=1, keepdims=True)) * chain", "P * dP * chain"),
    "bwd_dk_no_scale": ("dK[b, :, kh] += s * (dS.T @ Q[b, :, h])", "dK[b, :, kh] += dS.T @ Q[b, :, h]"),
    "bwd_dv_overwritten": ("dV[b, :, kh] += P.T @ dO[b, :, h]", "dV[b, :, kh] = P.T @ dO[b, :, h]"),
    "bwd_gqa_modulo": ("kh = h // G", "kh = h % Hk"),
    "bwd_dq_transposed_ds": ("dQ[b, :, h] = s * (dS @ K[b, :, kh])", "dQ[b, :, h] = s * (dS.T @ K[b, :, kh])"),
    "bwd_softcap_no_chain": ("chain = 1.0 - th * th", "chain = 1.0"),
    "bwd_alibi_sign": ("z = u - slopes[h] * dist", "z = u + slopes[h] * dist"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap

    src = textwrap.dedent(inspect.getsource(oracle.attention_bwd))
    a, b = BWD_MUTANTS[name]
    assert a in src, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(a, b), "<mutant>", "exec"), ns)
    monkeypatch.setattr(oracle, "attention_bwd", ns["attention_bwd"])
    with pytest.raises((AssertionError, ValueError, IndexError)):
        oracle_pins.pin_backward(oracle.load())


# Mistakes planted in the differential backward oracle.
DIFF_BWD_MUTANTS = {
    "diff_bwd_lambda_sign": ("coef = (1.0, -float(lam))", "coef = (1.0, float(lam))"),
    "diff_bwd_dv_one_stream": ("dV[b, :, kh] += coef[t] * (P.T @ dO[b, :, h])",
                               "dV[b, :, kh] += (P.T @ dO[b, :, h]) if t == 0 else 0.0"),
    "diff_bwd_streams_share_k": ("z = np.where(allowed, sc * (Q[t, b, :, h] @ K[t, b, :, kh].T), -np.inf)",
                                 "z = np.where(allowed, sc * (Q[t, b, :, h] @ K[0, b, :, kh].T), -np.inf)"),
    "diff_bwd_dk_from_other_q": ("dK[t, b, :, kh] += sc * (dS.T @ Q[t, b, :, h])",
                                 "dK[t, b, :, kh] += sc * (dS.T @ Q[1 - t, b, :, h])"),
    "diff_bwd_no_coef_in_dp": ("dP = coef[t] * (dO[b, :, h] @ V[b, :, kh].T)", "dP = dO[b, :, h] @ V[b, :, kh].T"),
}


@pytest.mark.parametrize("name", sorted(DIFF_BWD_MUTANTS))
def test_diff_bwd_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap

    src = textwrap.dedent(inspect.getsource(oracle.diff_attention_bwd))
    a, b = DIFF_BWD_MUTANTS[name]
    assert a in src, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(a, b), "<mutant>", "exec"), ns)
    monkeypatch.setattr(oracle, "diff_attention_bwd", ns["diff_attention_bwd"])
    with pytest.raises((AssertionError, ValueError, IndexError)):
        oracle_pins.pin_diff_backward(oracle.load())


ALLOWED_MUTANTS = {
    "allowed_window_inclusive": ("(i - j < window)", "(i - j <= window)"),
    "allowed_prefix_inclusive": ("(j < prefix)", "(j <= prefix)"),
    "allowed_doc_side_left": ('side="right"', 'side="left"'),
}


@pytest.mark.parametrize("name", sorted(ALLOWED_MUTANTS))
def test_allowed_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap

    src = textwrap.dedent(inspect.getsource(oracle._allowed))
    a, b = ALLOWED_MUTANTS[name]
    assert a in src, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(a, b), "<mutant>", "exec"), ns)
    monkeypatch.setattr(oracle, "_allowed", ns["_allowed"])
    with pytest.raises(AssertionError):
        oracle_pins.pin_backward(oracle.load())


# Mistakes planted in the oracle's forward-mode derivatives of expressions.
EXPR_GRAD_MUTANTS = {
    "grad_tanh_sign": ("return t, (1.0 - t * t) * da", "return t, (1.0 + t * t) * da"),
    "grad_div_sign": ("(da * b - a * db) / (b * b)", "(da * b + a * db) / (b * b)"),
    "grad_exp2_no_ln2": ("return e, e * ln2 * da", "return e, e * da"),
    "grad_min_picks_other": ("pick_a = (a <= b) if f == \"min\" else (a >= b)",
                             "pick_a = (a >= b) if f == \"min\" else (a >= b)"),
}


@pytest.mark.parametrize("name", sorted(EXPR_GRAD_MUTANTS))
def test_expr_grad_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap

    from oracle import score_expr as se

    src = textwrap.dedent(inspect.getsource(se.evaluate_with_grad))
    a, b = EXPR_GRAD_MUTANTS[name]
    assert a in src, name
    ns = dict(vars(se))
    exec(compile(src.replace(a, b), "<mutant>", "exec"), ns)
    monkeypatch.setattr(se, "evaluate_with_grad", ns["evaluate_with_grad"])
    with pytest.raises(AssertionError):
        oracle_pins.pin_backward_expr(oracle.load())


# Mistakes planted in the composed forms' sampled-row paths (the gate gather of
# the Evoformer passes, the order of the differential streams): the source of
# the one function is edited in memory and swapped in for the test.
COMPOSED_MUTANTS = {
    "evo_row_gate_axes_exchanged": ("evo_row", "gate[r[:, 0], r[:, 2], r[:, 1], :]",
                                    "gate[r[:, 0], r[:, 1], r[:, 2], :]"),
    "evo_row_gate_msa_row_from_head": ("evo_row", "gate[r[:, 0], r[:, 2], r[:, 1], :]",
                                       "gate[r[:, 1], r[:, 2], r[:, 1], :]"),
    "evo_col_gate_axes_exchanged": ("evo_col", "gt[r[:, 0], r[:, 2], r[:, 1], :]",
                                    "gt[r[:, 0], r[:, 1], r[:, 2], :]"),
    "evo_col_gate_not_swapped": ("evo_col", "gt[r[:, 0], r[:, 2], r[:, 1], :]",
                                 "gate[r[:, 0] % gate.shape[0], r[:, 2] % gate.shape[1], r[:, 1], :]"),
    "diff_streams_stacked_reversed": ("diff_attention", "np.stack([l1, l2])", "np.stack([l2, l1])"),
}


@pytest.mark.parametrize("name", sorted(COMPOSED_MUTANTS))
def test_composed_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap

    fn, a, b = COMPOSED_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn)))
    assert src.count(a) == 1, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(a, b), "<mutant>", "exec"), ns)
    monkeypatch.setattr(oracle, fn, ns[fn])
    with pytest.raises(AssertionError):
        oracle_pins.pin_composed_rows(oracle.load())
