"""GPU parity of attention against a KV cache (decode) with the oracle:
contiguous and paged caches, ragged cache lengths, one or several new tokens,
causal and softcap, and the serving workload at its full size."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import testdata
from testdata import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402

import attention_variant_gb300 as fa  # noqa: E402


def _inputs(tag, B, Sq, Hq, Hk, S):
    q = testdata.normal_bf16((B, Sq, Hq, 64), f"dec_{tag}", "q")
    k = testdata.normal_bf16((B, S, Hk, 64), f"dec_{tag}", "k")
    v = testdata.normal_bf16((B, S, Hk, 64), f"dec_{tag}", "v")
    return q, k, v


def _paged(tag, B, Sq, Hq, Hk, lens, page):
    """A paged cache: a pool of shuffled pages [n_pages, page, Hk, 64] (three
    spare pages of other data), the block table (entries past a sequence's
    last page are -1 and must never be read), and the same keys gathered into
    contiguous [B, S, Hk, 64] arrays for the oracle."""
    per = [-(-int(L) // page) for L in lens]
    n_pages = sum(per) + 3
    rng = np.random.default_rng(testdata.fnv1a64(f"dec_{tag}/pages") & 0xFFFFFFFF)
    perm = rng.permutation(n_pages).astype(np.int32)
    table = np.full((B, max(per)), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, : per[b]] = perm[at: at + per[b]]
        at += per[b]
    q = testdata.normal_bf16((B, Sq, Hq, 64), f"dec_{tag}", "q")
    kp = testdata.normal_bf16((n_pages, page, Hk, 64), f"dec_{tag}", "kpool")
    vp = testdata.normal_bf16((n_pages, page, Hk, 64), f"dec_{tag}", "vpool")
    S = max(per) * page
    k = np.zeros((B, S, Hk, 64), dtype=np.uint16)
    v = np.zeros((B, S, Hk, 64), dtype=np.uint16)
    for b in range(B):
        n = per[b] * page
        k[b, :n] = kp[table[b, : per[b]]].reshape(n, Hk, 64)
        v[b, :n] = vp[table[b, : per[b]]].reshape(n, Hk, 64)
    return q, kp, vp, table, k, v


def _run(q, kc, vc, lens, max_kv, *, table=None, mod="none", causal=True, calls=1):
    B, Sq, Hq, _ = q.shape
    qd, kd, vd = gu.dev(q), gu.dev(kc), gu.dev(vc)
    lens_t = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    table_t = torch.from_numpy(table).cuda() if table is not None else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = fa.make_decode_desc(lens_t, max_kv, score_mod=mod, softcap=20.0, causal=causal,
                            block_table=table_t, error_word=err)
    ws = torch.empty(fa.fl_attn_decode_workspace_size(qd, kd, d), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # the call must not depend on the workspace's contents
    results = []
    for _ in range(calls):
        out = torch.full((B, Sq, Hq, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
        fa.fl_attn_decode(qd, kd, vd, out, lse, d, ws)
        torch.cuda.synchronize()
        results.append((gu.f64(out), gu.f64(lse)))
    assert int(err.item()) == 0
    return results


def _ref(q, k, v, lens, mod, causal):
    return oracle.attention(q, k, v, mod=mod, softcap=20.0, mask="decode" if causal else "kv_len",
                            kv_len=np.asarray(lens, dtype=np.int32))


@pytest.mark.parametrize("Sq", [1, 4])
@pytest.mark.parametrize("mod,causal", [("none", True), ("softcap", True), ("none", False)])
def test_contiguous_cache(Sq, mod, causal):
    B, Hq, Hk, S = 3, 8, 2, 700
    q, k, v = _inputs(f"c{Sq}", B, Sq, Hq, Hk, S)
    lens = [700, 333, 5]
    (o, lse), = _run(q, k, v, lens, 700, mod=mod, causal=causal)
    oref, lref = _ref(q, k, v, lens, mod, causal)
    gu.compare(o, lse, oref, lref, what=f"decode contiguous Sq={Sq} {mod} causal={causal}")


@pytest.mark.parametrize("causal,lens", [(True, [100, 37, 1]), (False, [100, 37, 0])])
def test_cache_shorter_than_one_chunk(causal, lens):
    # the cache holds fewer keys than a chunk (a box of 100 rows), and an
    # empty cache (no causal mask: a row with no key gives O = 0, LSE = -inf)
    B, Sq, Hq, Hk, S = 3, 1, 8, 2, 100
    q, k, v = _inputs(f"short{int(causal)}", B, Sq, Hq, Hk, S)
    (o, lse), = _run(q, k, v, lens, S, causal=causal)
    oref, lref = _ref(q, k, v, lens, "none", causal)
    gu.compare(o, lse, oref, lref, what=f"decode short cache causal={causal}")


@pytest.mark.parametrize("page", [16, 64, 256])
def test_paged_cache(page):
    B, Sq, Hq, Hk = 4, 2, 8, 2
    lens = [1100, 257, 256, 3]
    q, kp, vp, table, k, v = _paged(f"p{page}", B, Sq, Hq, Hk, lens, page)
    (o, lse), = _run(q, kp, vp, lens, max(lens), table=table, mod="softcap")
    oref, lref = _ref(q, k, v, lens, "softcap", True)
    gu.compare(o, lse, oref, lref, what=f"decode paged page={page}")


@pytest.mark.parametrize("Hq,Hk,Sq", [(32, 2, 2), (6, 2, 7), (16, 2, 5), (32, 2, 4)])
def test_many_query_rows(Hq, Hk, Sq):
    # G * Sq query rows per KV head: 32, 21, 40 and 64 (two to four groups
    # of 16 rows, the last one ragged or empty)
    B, S = 2, 450
    q, k, v = _inputs(f"rows{Hq}_{Sq}", B, Sq, Hq, Hk, S)
    lens = [450, 200]
    for mod in ("none", "softcap"):
        (o, lse), = _run(q, k, v, lens, S, mod=mod)
        oref, lref = _ref(q, k, v, lens, mod, True)
        gu.compare(o, lse, oref, lref, what=f"decode rows={Hq // Hk * Sq} {mod}")


def test_splits_of_several_chunks():
    # 256 sequences x 1 KV head with caches of up to 4096 keys: splits of 512
    # keys (four chunks, so the three-stage ring wraps), ragged last splits
    B, Sq, Hq, Hk, S = 256, 2, 4, 1, 4096
    q, k, v = _inputs("splits", B, Sq, Hq, Hk, S)
    lens = testdata.kv_lengths(B, "dec_splits", Sq, S)
    for causal in (True, False):
        (o, lse), = _run(q, k, v, lens, S, causal=causal)
        oref, lref = _ref(q, k, v, lens, "none", causal)
        gu.compare(o, lse, oref, lref, what=f"decode splits causal={causal}")


def test_two_calls_share_one_workspace():
    B, Sq, Hq, Hk, S = 2, 1, 4, 1, 600
    q, k, v = _inputs("twice", B, Sq, Hq, Hk, S)
    lens = [600, 513]
    (o1, l1), (o2, l2) = _run(q, k, v, lens, 600, calls=2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    oref, lref = _ref(q, k, v, lens, "none", True)
    gu.compare(o1, l1, oref, lref, what="decode first call")


def test_serving_workload_full_size():
    w = workloads.DECODE
    B, Sq, Hq, Hk = w["B"], w["Sq"], w["Hq"], w["Hk"]
    lens = testdata.kv_lengths(B, w["name"], w["kv_lo"], w["kv_hi"])
    q, kp, vp, table, k, v = _paged("serving", B, Sq, Hq, Hk, lens, w["page"])
    for mod in ("none", "softcap"):
        (o, lse), = _run(q, kp, vp, lens, int(lens.max()), table=table, mod=mod)
        oref, lref = _ref(q, k, v, lens, mod, True)
        gu.compare(o, lse, oref, lref, what=f"decode serving {mod}")
