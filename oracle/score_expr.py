"""Oracle for attention with a score_mod expression -- TEST INFRASTRUCTURE ONLY.

The Flashlight pages' generic-variant interface: a variant is an elementwise
expression over the scaled score and its indices, fused into the attention
(talk notes, "Compiler design" and the comparison with FlexAttention's
score_mod).  Here the expression is a string in the grammar of
``include/fl_attn.h`` (FL_MOD_EXPR); this module evaluates it on the full
``[Sq, Sk]`` score matrix of every (batch, head) in float64 with numpy, then
takes the plain two-pass softmax and ``P V``.  It shares no code with the CUDA
library, which translates the same string to CUDA on its own.

The string is parsed with Python's ``ast`` and only the grammar's node kinds
are evaluated (numbers, the five variables, ``inf``, the listed functions,
``+ - * /``, unary sign, one comparison): Python and the grammar agree on the
meaning and precedence of exactly that subset.
"""
from __future__ import annotations

import ast

import numpy as np

_VARS = ("score", "b", "h", "q_idx", "kv_idx")
_FUNCS = {
    "tanh": (1, np.tanh), "exp": (1, np.exp), "exp2": (1, np.exp2), "log": (1, np.log),
    "log2": (1, np.log2), "sqrt": (1, np.sqrt), "abs": (1, np.abs), "floor": (1, np.floor),
    "min": (2, np.minimum), "max": (2, np.maximum),
    "where": (3, lambda c, x, y: np.where(np.asarray(c) != 0, x, y)),
}
_BIN = {ast.Add: np.add, ast.Sub: np.subtract, ast.Mult: np.multiply, ast.Div: np.divide}
_CMP = {ast.Lt: np.less, ast.LtE: np.less_equal, ast.Gt: np.greater,
        ast.GtE: np.greater_equal, ast.Eq: np.equal, ast.NotEq: np.not_equal}


def parse(expr: str) -> ast.Expression:
    """Parse and check ``expr`` against the grammar; raises ValueError."""
    try:
        tree = ast.parse(expr, mode="eval")
    except SyntaxError as e:
        raise ValueError(f"not an expression: {e.msg}") from None
    for node in ast.walk(tree):
        ok = isinstance(node, (ast.Expression, ast.BinOp, ast.UnaryOp, ast.Compare, ast.Call,
                               ast.Name, ast.Constant, ast.Load)) or type(node) in _BIN \
            or type(node) in _CMP or isinstance(node, (ast.USub, ast.UAdd))
        if not ok:
            raise ValueError(f"{type(node).__name__} is not part of the grammar")
        if isinstance(node, ast.BinOp) and type(node.op) not in _BIN:
            raise ValueError("operator not part of the grammar")
        if isinstance(node, ast.Compare) and len(node.ops) != 1:
            raise ValueError("comparisons do not chain")
        if isinstance(node, ast.Constant) and (isinstance(node.value, bool)
                                               or not isinstance(node.value, (int, float))):
            raise ValueError("only numbers are constants")
        if isinstance(node, ast.Call):
            if not isinstance(node.func, ast.Name) or node.func.id not in _FUNCS or node.keywords:
                raise ValueError("unknown function")
            if len(node.args) != _FUNCS[node.func.id][0]:
                raise ValueError(f"{node.func.id} takes {_FUNCS[node.func.id][0]} arguments")
        if isinstance(node, ast.Name) and node.id not in _VARS + ("inf",) + tuple(_FUNCS):
            raise ValueError(f"unknown name {node.id}")
    called = {id(n.func) for n in ast.walk(tree) if isinstance(n, ast.Call)}
    for node in ast.walk(tree):
        if isinstance(node, ast.Name) and node.id in _FUNCS and id(node) not in called:
            raise ValueError(f"{node.id} is a function")
    return tree


def evaluate(expr: str, **env) -> np.ndarray:
    """Value of ``expr`` with the variables in ``env`` (float64 arrays or
    scalars that broadcast); comparisons give 1.0 or 0.0."""
    tree = parse(expr)

    def ev(n):
        if isinstance(n, ast.Expression):
            return ev(n.body)
        if isinstance(n, ast.Constant):
            return np.float64(n.value)
        if isinstance(n, ast.Name):
            return np.float64(np.inf) if n.id == "inf" else np.asarray(env[n.id], dtype=np.float64)
        if isinstance(n, ast.UnaryOp):
            x = ev(n.operand)
            return -x if isinstance(n.op, ast.USub) else x
        if isinstance(n, ast.BinOp):
            return _BIN[type(n.op)](ev(n.left), ev(n.right))
        if isinstance(n, ast.Compare):
            return _CMP[type(n.ops[0])](ev(n.left), ev(n.comparators[0])).astype(np.float64)
        if isinstance(n, ast.Call):
            return _FUNCS[n.func.id][1](*[ev(a) for a in n.args])
        raise ValueError(type(n).__name__)

    with np.errstate(all="ignore"):
        return ev(tree)


def evaluate_with_grad(expr: str, **env):
    """Value of ``expr`` and its derivative with respect to ``score``
    (forward-mode differentiation: every node carries (value, derivative)),
    float64.  Comparisons, ``floor`` and the condition of ``where`` are
    piecewise constant (derivative 0); ``abs`` takes the derivative +1 at 0."""
    tree = parse(expr)
    ln2 = np.log(2.0)

    def ev(n):
        if isinstance(n, ast.Expression):
            return ev(n.body)
        if isinstance(n, ast.Constant):
            return np.float64(n.value), np.float64(0.0)
        if isinstance(n, ast.Name):
            if n.id == "inf":
                return np.float64(np.inf), np.float64(0.0)
            x = np.asarray(env[n.id], dtype=np.float64)
            return x, (np.ones_like(x) if n.id == "score" else np.zeros_like(x))
        if isinstance(n, ast.UnaryOp):
            v, d = ev(n.operand)
            return (-v, -d) if isinstance(n.op, ast.USub) else (v, d)
        if isinstance(n, ast.BinOp):
            (a, da), (b, db) = ev(n.left), ev(n.right)
            if isinstance(n.op, ast.Add):
                return a + b, da + db
            if isinstance(n.op, ast.Sub):
                return a - b, da - db
            if isinstance(n.op, ast.Mult):
                return a * b, da * b + a * db
            return a / b, (da * b - a * db) / (b * b)
        if isinstance(n, ast.Compare):
            (a, _), (b, _) = ev(n.left), ev(n.comparators[0])
            v = _CMP[type(n.ops[0])](a, b).astype(np.float64)
            return v, np.zeros_like(v)
        if isinstance(n, ast.Call):
            args = [ev(x) for x in n.args]
            f = n.func.id
            (a, da) = args[0]
            if f == "tanh":
                t = np.tanh(a)
                return t, (1.0 - t * t) * da
            if f == "exp":
                e = np.exp(a)
                return e, e * da
            if f == "exp2":
                e = np.exp2(a)
                return e, e * ln2 * da
            if f == "log":
                return np.log(a), da / a
            if f == "log2":
                return np.log2(a), da / (a * ln2)
            if f == "sqrt":
                r = np.sqrt(a)
                return r, da / (2.0 * r)
            if f == "abs":
                return np.abs(a), np.where(a >= 0, da, -da)
            if f == "floor":
                return np.floor(a), np.zeros_like(np.asarray(a, dtype=np.float64))
            if f in ("min", "max"):
                (b, db) = args[1]
                pick_a = (a <= b) if f == "min" else (a >= b)
                return (np.minimum(a, b) if f == "min" else np.maximum(a, b)), np.where(pick_a, da, db)
            (x, dx), (y, dy) = args[1], args[2]   # where(c, x, y)
            c = np.asarray(a) != 0
            return np.where(c, x, y), np.where(c, dx, dy)
        raise ValueError(type(n).__name__)

    with np.errstate(all="ignore"):
        return ev(tree)


def _widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention_expr(q, k, v, expr: str, *, mask="none", scale=0.0):
    """Attention with the logits ``expr`` (over score = scale q.k, b, h, q_idx,
    kv_idx) of ``q [B,S,Hq,D]``, ``k [B,S,Hk,D]``, ``v [B,S,Hk,Dv]`` (bf16
    bits), with the ``none`` or ``causal`` mask on top.  Returns float64
    ``O [B,S,Hq,Dv]`` and natural-log ``LSE [B,Hq,S]``; a row with no
    allowed key gives O = 0 and LSE = -inf."""
    if mask not in ("none", "causal"):
        raise ValueError("mask must be none or causal")
    parse(expr)
    qf, kf, vf = _widen(q), _widen(k), _widen(v)
    B, S, Hq, D = qf.shape
    Hk = kf.shape[2]
    G = Hq // Hk
    s = scale if scale else 1.0 / np.sqrt(D)
    i = np.arange(S, dtype=np.float64)[:, None]
    j = np.arange(kf.shape[1], dtype=np.float64)[None, :]
    out = np.zeros((B, S, Hq, vf.shape[3]))
    lse = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            score = s * (qf[b, :, h, :] @ kf[b, :, h // G, :].T)
            z = np.broadcast_to(evaluate(expr, score=score, b=float(b), h=float(h), q_idx=i,
                                         kv_idx=j), score.shape).copy()
            if mask == "causal":
                z[j > i] = -np.inf
            m = z.max(axis=1, keepdims=True)
            empty = ~np.isfinite(m[:, 0]) & (m[:, 0] < 0)
            m[empty] = 0.0
            with np.errstate(all="ignore"):
                p = np.exp(z - m)
            l = p.sum(axis=1)
            o = p @ vf[b, :, h // G, :]
            with np.errstate(divide="ignore", invalid="ignore"):
                out[b, :, h, :] = np.where(l[:, None] > 0, o / l[:, None], 0.0)
                lse[b, h, :] = np.where(l > 0, m[:, 0] + np.log(l), -np.inf)
    return out, lse
