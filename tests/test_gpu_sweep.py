"""Seeded random sweep of shapes and variants for every forward kind, each
compared with the oracle over the whole output (and its visited-tile counts).

The fixed-shape tests choose their cases by hand; this sweep draws batch,
length, head counts, head dimensions, masks, score_mods and lambda at random
(seeded, so every run sees the same cases) to reach combinations nobody
picked.  Within the bf16 limits of the 1e-2 O bound (ALiBi and softcap at
D <= 64, documents of at least 37 keys), every case must meet the same
tolerances as the fixed-shape tests.
"""
import numpy as np
import pytest
import torch

import attention_variant_gb300 as fa
import oracle
import testdata
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

SEED = 20261220  # chosen so the draw covers every head dimension, mask and score_mod


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_variant_gb300 import build
    build.build()


def _std_cases(n=24):
    rng = np.random.default_rng(SEED)
    cases = []
    for c in range(n):
        D = int(rng.choice([32, 64, 128]))
        Hk = int(rng.choice([1, 2]))
        Hq = Hk * int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 4))
        S = int(rng.integers(1, 1400))
        mask = str(rng.choice(["none", "causal", "window", "prefix", "doc"]))
        mod = str(rng.choice(["none", "alibi", "softcap"])) if D <= 64 else "none"
        kw = {}
        if mask == "window":
            kw["window"] = int(rng.integers(1, S + 50))
        elif mask == "prefix":
            kw["prefix"] = int(rng.integers(0, S + 50))
        cases.append((c, B, S, Hq, Hk, D, mask, mod, kw))
    return cases


@pytest.mark.parametrize("case", _std_cases(), ids=lambda c: f"std{c[0]}")
def test_sweep_standard(case):
    c, B, S, Hq, Hk, D, mask, mod, kw = case
    tag = f"sweep_std{c}"
    q = testdata.normal_bf16((B, S, Hq, D), tag, "q")
    k = testdata.normal_bf16((B, S, Hk, D), tag, "k")
    v = testdata.normal_bf16((B, S, Hk, D), tag, "v")
    if mask == "doc":
        kw = dict(doc_offsets=testdata.doc_offsets(S, B, tag, lo=37, hi=400))
    o, lse, cnt, err = gu.run_standard(q, k, v, score_mod=mod, mask=mask, softcap=20.0, **dict(kw))
    assert err == 0
    oref, lref = oracle.attention(q, k, v, mod=mod, mask=mask, softcap=20.0, **kw)
    gu.compare(o, lse, oref, lref, what=f"{tag}: B{B} S{S} H{Hq}/{Hk} D{D} {mod}/{mask} {kw}")
    bn = fa.fl_attn_tile_shape(fa.make_desc(), D)[1]
    exp = gu.expected_tile_counts(mask, B, Hq, S, kw.get("window", 0), kw.get("prefix", 0),
                                  kw.get("doc_offsets"), bn=bn)
    assert np.array_equal(cnt, exp), f"{tag}: tile counts differ"


def _diff_cases(n=8):
    rng = np.random.default_rng(SEED + 1)
    return [(c, int(rng.integers(1, 4)), int(rng.integers(1, 1200)), int(rng.choice([1, 2])),
             int(rng.choice([1, 2, 3])), int(rng.choice([64, 128])), str(rng.choice(["none", "causal"])),
             float(rng.uniform(-1.0, 1.0))) for c in range(n)]


@pytest.mark.parametrize("case", _diff_cases(), ids=lambda c: f"diff{c[0]}")
def test_sweep_diff(case):
    c, B, S, Hk, G, Dv, mask, lam = case
    H = Hk * G
    tag = f"sweep_diff{c}"
    q = testdata.normal_bf16((2, B, S, H, 64), tag, "q")
    k = testdata.normal_bf16((2, B, S, Hk, 64), tag, "k")
    v = testdata.normal_bf16((B, S, Hk, Dv), tag, "v")
    out = torch.full((B, S, H, Dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((2, B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    cnt = torch.full((B, H, (S + 127) // 128), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = fa.make_desc(kind="diff", mask=mask, diff_lambda=lam, debug_tile_counts=cnt, error_word=err)
    fa.fl_attn_fwd(gu.dev(q), gu.dev(k), gu.dev(v), out, lse, d)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oref, lref = oracle.diff_attention(q, k, v, lam, mask=mask)
    gu.compare(gu.f64(out), gu.f64(lse), oref, lref, what=f"{tag}: B{B} S{S} H{H}/{Hk} Dv{Dv} {mask} lam {lam:.3f}")
    bn = fa.fl_attn_tile_shape(fa.make_desc(kind="diff"), Dv)[1]
    assert np.array_equal(cnt.cpu().numpy(), gu.expected_tile_counts(mask, B, H, S, bn=bn))


def _evo_cases(n=8):
    rng = np.random.default_rng(SEED + 2)
    cases = []
    for c in range(n):
        row = bool(rng.integers(0, 2))
        Ns = int(rng.integers(1, 300))
        Nr = 8 * int(rng.integers(1, 70)) if row else int(rng.integers(1, 40))  # bias rows: 16-byte pitch
        cases.append((c, row, Ns, Nr, int(rng.integers(1, 5)), int(rng.choice([32, 64]))))
    return cases


@pytest.mark.parametrize("case", _evo_cases(), ids=lambda c: f"evo{c[0]}")
def test_sweep_evoformer(case):
    c, row, Ns, Nr, H, ch = case
    tag = f"sweep_evo{c}"
    q, k, v, g = (testdata.normal_bf16((Ns, Nr, H, ch), tag, n) for n in ("q", "k", "v", "g"))
    bias = testdata.normal_bf16((H, Nr, Nr), tag, "bias") if row else None
    B, S = (Ns, Nr) if row else (Nr, Ns)
    out = torch.full((Ns, Nr, H, ch), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    cnt = torch.full((B, H, (S + 127) // 128), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = fa.make_desc(kind="evo_row" if row else "evo_col", debug_tile_counts=cnt, error_word=err)
    fa.fl_attn_fwd(gu.dev(q), gu.dev(k), gu.dev(v), out, lse, d, bias=gu.dev(bias) if row else None,
                   gate=gu.dev(g))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    if row:
        oref, lref = oracle.evo_row(q, k, v, bias, g)
    else:
        oref, lref = oracle.evo_col(q, k, v, g)
        oref = np.swapaxes(oref, 0, 1)
    gu.compare(gu.f64(out), gu.f64(lse), oref, lref,
               what=f"{tag}: {'row' if row else 'col'} Ns{Ns} Nr{Nr} H{H} c{ch}")
    bn = fa.fl_attn_tile_shape(fa.make_desc(kind="evo_row"), ch)[1]
    assert np.array_equal(cnt.cpu().numpy(), gu.expected_tile_counts("none", B, H, S, bn=bn))


def _decode_cases(n=8):
    rng = np.random.default_rng(SEED + 3)
    cases = []
    for c in range(n):
        Sq = int(rng.integers(1, 5))
        Hk = int(rng.choice([1, 2]))
        G = int(rng.choice([g for g in (1, 2, 4, 8) if g * Sq <= 64]))
        B = int(rng.integers(1, 9))
        lens = [int(x) for x in rng.integers(Sq, 3000, size=B)]
        page = int(rng.choice([0, 16, 64, 256]))  # 0: contiguous cache
        cases.append((c, B, Sq, Hk * G, Hk, lens, page, str(rng.choice(["none", "softcap"])),
                      bool(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("case", _decode_cases(), ids=lambda c: f"decode{c[0]}")
def test_sweep_decode(case):
    from tests import test_gpu_decode as td

    c, B, Sq, Hq, Hk, lens, page, mod, causal = case
    tag = f"sweep_dec{c}"
    if page:
        q, kc, vc, table, k, v = td._paged(tag, B, Sq, Hq, Hk, lens, page)
    else:
        q, k, v = td._inputs(tag, B, Sq, Hq, Hk, max(lens))
        kc, vc, table = k, v, None
    (o, lse), = td._run(q, kc, vc, lens, max(lens), table=table, mod=mod, causal=causal)
    oref, lref = td._ref(q, k, v, lens, mod, causal)
    gu.compare(o, lse, oref, lref, what=f"{tag}: B{B} Sq{Sq} H{Hq}/{Hk} page {page} {mod} causal={causal}")


def _bwd_cases(n=6):
    rng = np.random.default_rng(SEED + 4)
    cases = []
    for c in range(n):
        Hk = int(rng.choice([1, 2]))
        Hq = Hk * int(rng.choice([1, 2, 4]))
        S = int(rng.integers(1, 700))
        mask = str(rng.choice(["none", "causal", "window", "prefix", "doc"]))
        kw = {}
        if mask == "window":
            kw["window"] = int(rng.integers(1, S + 50))
        elif mask == "prefix":
            kw["prefix"] = int(rng.integers(0, S + 50))
        cases.append((c, int(rng.integers(1, 3)), S, Hq, Hk, mask, str(rng.choice(["none", "alibi", "softcap"])),
                      kw))
    return cases


@pytest.mark.parametrize("case", _bwd_cases(), ids=lambda c: f"bwd{c[0]}")
def test_sweep_backward(case):
    from tests import test_gpu_bwd as tb

    c, B, S, Hq, Hk, mask, mod, kw = case
    tag = f"sweep_bwd{c}"
    if mask == "doc":
        kw = dict(doc_offsets=testdata.doc_offsets(S, B, tag, lo=37, hi=400))
    got, ref = tb._run(tag, B, S, Hq, Hk, mask, mod=mod, **kw)
    tb._check(got, ref, f"{tag}: B{B} S{S} H{Hq}/{Hk} {mod}/{mask}")


def _diff_bwd_cases(n=4):
    rng = np.random.default_rng(SEED + 5)
    return [(c, int(rng.integers(1, 3)), int(rng.integers(1, 600)), int(rng.choice([1, 2])),
             int(rng.choice([1, 2, 3])), int(rng.choice([64, 128])), str(rng.choice(["none", "causal"])),
             float(rng.uniform(-1.0, 1.0))) for c in range(n)]


@pytest.mark.parametrize("case", _diff_bwd_cases(), ids=lambda c: f"diffbwd{c[0]}")
def test_sweep_diff_backward(case):
    from tests import test_gpu_diff_bwd as tdb

    c, B, S, Hk, G, Dv, mask, lam = case
    got, ref = tdb._run(f"sweep{c}", B, S, Hk * G, Hk, Dv, mask, lam)
    tdb._check(got, ref, f"sweep diff backward {c}: B{B} S{S} H{Hk * G}/{Hk} Dv{Dv} {mask} lam {lam:.3f}")
