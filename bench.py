#!/usr/bin/env python
"""Fused attention forward throughput on GB300: TFLOP/s and fraction of peak.

Headline workload: the MHA score_mod sweep at S = 2048 (B = 8, H = 16, D = 64,
bf16 inputs drawn N(0,1) from the shared seeded generator), vanilla
non-causal.  A step is one fused forward (O and LSE) over that batch, with the
inputs already resident in HBM.  L2 is flushed (a 256 MiB write) before every
timed step, and each step is timed with CUDA events on the launching stream.
Variant workloads whose bytes exceed twice the L2 (the Evoformer, differential
and KV-cache decode ones) run back to back without the flush, each variant
record saying which.

Flops are algorithmic: 4 * D per unmasked (query, key) pair.  The per-variant
table ("variants") repeats the measurement for every variant and sequence
length of the MHA sweep and the GQA mask sweep.

--impl reference times the CPU oracle (the plain double-precision definition)
on the host cores on a bounded sample of the same workload.

For N > 1 (torchrun), every rank runs the same per-GPU workload on its own
GPU with no collective on the data path (independent shards: weak scaling);
value = all ranks' flops / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import testdata  # noqa: E402
from testdata import workloads  # noqa: E402

HEADLINE = dict(S=2048, variant="vanilla")
METRIC = "fused attention fwd TFLOP/s (bf16) and % of GB300 dense BF16 peak per variant"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20  # GB300 L2


def l2_policy(e):
    """Workloads whose bytes exceed twice the L2 run back to back unflushed
    (their inputs cannot stay in L2 between steps); a flush would also leave
    256 MiB of dirty lines for the timed kernel to write back."""
    return "unflushed: inputs larger than L2" if e["bytes"] > 2 * L2_BYTES else \
        "flushed before every timed step (256 MiB write)"
KERNEL_SOURCES = ["attention_variant_gb300/csrc/fwd_standard.cu",
                  "attention_variant_gb300/csrc/softmax_tile.cuh",
                  "attention_variant_gb300/csrc/common.cuh",
                  "attention_variant_gb300/csrc/ptx.cuh",
                  "attention_variant_gb300/csrc/fastdiv.h"]


# ---------------------------------------------------------------- workload accounting

def row_intervals(mask, S, window=0, prefix=0, starts=None):
    """Allowed keys [lo_i, hi_i) of every query row (the masks' definitions)."""
    i = np.arange(S, dtype=np.int64)
    if mask == "none":
        return np.zeros(S, np.int64), np.full(S, S, np.int64)
    if mask == "causal":
        return np.zeros(S, np.int64), i + 1
    if mask == "window":
        return np.maximum(0, i - window + 1), i + 1
    if mask == "prefix":
        return np.zeros(S, np.int64), np.minimum(S, np.maximum(i + 1, prefix))
    if mask == "doc":
        st = np.asarray(starts)
        st = st[st < S]
        ds = st[np.searchsorted(st, i, side="right") - 1]
        return ds, i + 1
    raise ValueError(mask)


def unmasked_pairs(mask, B, H, S, window=0, prefix=0, doc=None):
    total = 0
    for b in range(B):
        lo, hi = row_intervals(mask, S, window, prefix, None if doc is None else doc[b])
        total += int((hi - lo).sum()) * H
    return total


def visited_pairs(mask, B, H, S, bn, window=0, prefix=0, doc=None):
    """Pairs inside the key tiles the kernel visits: per 128-row query block,
    its rows times the keys of the tiles [floor(lo_first / bn), ceil(hi_last / bn))
    (the last tile clipped to S).  Against the unmasked pairs it shows the
    work spent on masked pairs of partial tiles."""
    total = 0
    for b in range(B):
        lo, hi = row_intervals(mask, S, window, prefix, None if doc is None else doc[b])
        q0 = np.arange(0, S, 128)
        q1 = np.minimum(q0 + 128, S)
        t_lo = lo[q0] // bn
        t_hi = -(-hi[q1 - 1] // bn)
        keys = np.minimum(t_hi * bn, S) - t_lo * bn
        total += int(((q1 - q0) * keys).sum()) * H
    return total


# XU-pipe cycles per visited pair and sub-partition: a 2^x takes 4 cycles per
# warp instruction (32 pairs), the bf16 pack of two P 2 cycles; softcap adds a
# 2^x and a reciprocal (probed rates, 32 2^x per clock and SM).
XU_CYCLES_PER_PAIR = {"none": (4 + 1) / 32, "alibi": (4 + 1) / 32, "softcap": (12 + 1) / 32}


def bound_times(e, peaks, sms=152, clock_hz=2.07e9):
    """The launch's lower bounds in us: tensor (algorithmic flops at the
    measured bf16 peak), HBM (algorithmic bytes at the measured copy rate) and
    XU (the special-function work of the visited pairs at the maximum clock)."""
    out = dict(t_tc_us=round(e["flops"] / (peaks["bf16_tflops"] * 1e12) * 1e6, 1),
               t_hbm_us=round(e["bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e6, 1))
    if "visited" in e:
        xu = e["visited"] * XU_CYCLES_PER_PAIR.get(e.get("mod", "none"), XU_CYCLES_PER_PAIR["none"])
        out["t_xu_us"] = round(xu / (4 * sms * clock_hz) * 1e6, 1)
    return out


VARIANT_WARMUP = 3  # untimed launches before each variant's timed steps


def spread(ms):
    """Median and standard deviation of per-step times (the mean is the value)."""
    return dict(median_ms=round(statistics.median(ms), 4),
                std_ms=round(statistics.pstdev(ms), 4) if len(ms) > 1 else 0.0)


def entry(kind, S, variant, D=workloads.HEAD_DIM):
    """One benchmark entry of the MHA sweep ("mha") or GQA mask sweep ("gqa");
    D other than the sweep's 64 names a head-dimension variant of its shape."""
    if kind == "mha":
        w = workloads.mha_workload(S)
        B, Hq, Hk = w["B"], w["H"], w["H"]
    else:
        B = dict(workloads.GQA_SHAPES)[S]
        w = workloads.gqa_workload(S, B)
        Hq, Hk = w["Hq"], w["Hk"]
    if D != workloads.HEAD_DIM:
        w = dict(w, name=f"{w['name']}_d{D}")
    mod = {"vanilla": "none", "alibi": "alibi", "softcap": "softcap"}.get(variant, "none")
    mask = variant if variant in ("causal", "window", "prefix", "doc") else "none"
    kw = {}
    doc = None
    if mask == "window":
        kw["window"] = workloads.WINDOW
    elif mask == "prefix":
        kw["prefix"] = workloads.PREFIX
    elif mask == "doc":
        doc = testdata.doc_offsets(S, B, w["name"], *workloads.DOC_LEN_RANGE)
    pairs = unmasked_pairs(mask, B, Hq, S, kw.get("window", 0), kw.get("prefix", 0), doc)
    return dict(name=w["name"], kind=kind, B=B, Hq=Hq, Hk=Hk, S=S, D=D, variant=variant,
                mod=mod, mask=mask, kw=kw, doc=doc, pairs=pairs, flops=4 * D * pairs,
                bytes=2 * B * S * D * (2 * Hq + 2 * Hk) + 4 * B * Hq * S)


# Score_mod expressions compiled at run time, on the same workload as the
# built-in variant each one restates (the pages' generic-variant interface).
EXPR_VARIANTS = {
    "expr_softcap": ("softcap", "20 * tanh(score / 20)"),
    "expr_alibi": ("alibi", "score - exp2(-8 * (h + 1) / 16) * abs(q_idx - kv_idx)"),
}


def expr_entry(S, name):
    builtin, expr = EXPR_VARIANTS[name]
    e = entry("mha", S, builtin)
    e.update(variant=name, mod="expr", kw={"score_expr": expr})
    return e


def diff_entry(mask, Dv=None):
    w = workloads.DIFF
    B, S, H, D = w["B"], w["S"], w["H"], w["D"]
    Dv = Dv or w["Dv"]
    name = w["name"] if Dv == w["Dv"] else f"{w['name']}_dv{Dv}"
    pairs = unmasked_pairs(mask, B, H, S)
    # per pair: two Q K^T (2 D each) and two P V (2 Dv each)
    return dict(name=name, kind="diff", B=B, S=S, H=H, D=D, Dv=Dv, mask=mask,
                variant="causal" if mask == "causal" else "non-causal", pairs=pairs,
                flops=pairs * (2 * 2 * D + 2 * 2 * Dv),
                bytes=2 * (2 * 2 * B * S * H * D + B * S * H * Dv + B * S * H * Dv) + 4 * 2 * B * H * S)


def evo_entry(row, w=None):
    w = w or workloads.EVO
    Ns, Nr, H, c = w["N_seq"], w["N_res"], w["H"], w["c"]
    B, S = (Ns, Nr) if row else (Nr, Ns)
    pairs = B * H * S * S
    tensor_bytes = Ns * Nr * H * c * 2
    return dict(name=w["name"], kind="evo_row" if row else "evo_col", variant="row" if row else "col",
                Ns=Ns, Nr=Nr, H=H, c=c, pairs=pairs, flops=pairs * 4 * c,
                bytes=5 * tensor_bytes + (H * Nr * Nr * 2 if row else 0))


def evo_batched_entry(row):
    """A batch of MSA stacks with an MSA mask, through fl_attn_evoformer."""
    w = workloads.EVO_AF2
    Bt, Ns, Nr, H, c = w["B"], w["N_seq"], w["N_res"], w["H"], w["c"]
    mask = np.ones((Bt, Ns, Nr), dtype=np.float32)
    mask[:, :, Nr - w["pad_res"]:] = 0.0  # padding residues
    mask[:, Ns - w["pad_seq"]:, :] = 0.0  # padding MSA rows
    kept = mask.sum(axis=2) if row else mask.sum(axis=1)  # keys per (stack, batch index)
    q_rows = Nr if row else Ns
    pairs = int(kept.sum()) * H * q_rows
    tensor_bytes = Bt * Ns * Nr * H * c * 2
    return dict(name=w["name"], kind="evo_batched", row=row, variant="row_masked" if row else "col_masked",
                Bt=Bt, Ns=Ns, Nr=Nr, H=H, c=c, mask=mask, pairs=pairs, flops=pairs * 4 * c,
                bytes=5 * tensor_bytes + (Bt * H * Nr * Nr * 2 if row else 0) + mask.size * 4)


def bwd_entry(mask, expr=None, mod="none"):
    """The backward (dQ, dK, dV) on the headline MHA workload; algorithmic
    flops 10 D per unmasked pair (the five products of the gradient).  With
    ``expr`` the score_mod is that run-time expression."""
    e = entry("mha", HEADLINE["S"], "causal" if mask == "causal" else "vanilla")
    name = ("bwd_expr_softcap" if expr is not None else "bwd_softcap" if mod == "softcap"
            else "bwd_" + ("causal" if mask == "causal" else "vanilla"))
    e.update(kind="bwd", variant=name, expr=expr, mod=mod,
             flops=10 * e["D"] * e["pairs"],
             bytes=2 * e["B"] * e["S"] * e["D"] * (4 * e["Hq"] + 4 * e["Hk"]) + 4 * e["B"] * e["Hq"] * e["S"])
    return e


def time_bwd(e, torch, fa, device, steps, warmup, flush, stream):
    """Device time of fl_attn_bwd (its three launches) on the workload."""
    B, S, Hq, Hk, D = e["B"], e["S"], e["Hq"], e["Hk"], e["D"]
    q, k, v = gpu_inputs(e, torch, device)
    q, k, v = q.to(device), k.to(device), v.to(device)
    do = torch.from_numpy(testdata.normal_bf16((B, S, Hq, D), e["name"], "do").view(np.int16)) \
        .view(torch.bfloat16).to(device)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=device)
    desc = fa.make_desc(mask=e["mask"], score_mod=e["mod"], softcap=workloads.SOFTCAP, score_expr=e.get("expr"))
    fa.fl_attn_fwd(q, k, v, out, lse, desc)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fl_attn_bwd_workspace_size(q, k, desc), dtype=torch.uint8, device=device)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            fa.fl_attn_bwd(q, k, v, out, lse, do, dq, dk, dv, desc, ws, stream=stream)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fa.fl_attn_bwd(q, k, v, out, lse, do, dq, dk, dv, desc, ws, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def diff_bwd_entry(mask):
    """The differential backward on the differential workload; algorithmic
    flops per unmasked pair and stream 6 D + 4 Dv (S = Q K^T, dQ and dK: 2 D
    each; dP = dO V^T and dV: 2 Dv each)."""
    e = diff_entry(mask)
    e.update(kind="diff_bwd", variant="bwd_" + ("causal" if mask == "causal" else "non-causal"),
             flops=e["pairs"] * 2 * (6 * e["D"] + 4 * e["Dv"]),
             bytes=2 * e["B"] * e["S"] * e["H"] * (2 * 2 * 2 * e["D"] + 3 * e["Dv"]) + 4 * 2 * e["B"] * e["H"] * e["S"])
    return e


def time_diff_bwd(e, torch, fa, device, steps, warmup, flush, stream):
    """Device time of fl_attn_diff_bwd (all its launches) on the workload."""
    B, S, H, D, Dv = e["B"], e["S"], e["H"], e["D"], e["Dv"]
    to = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(device)
    q = to(testdata.normal_bf16((2, B, S, H, D), e["name"], "q"))
    k = to(testdata.normal_bf16((2, B, S, H, D), e["name"], "k"))
    v = to(testdata.normal_bf16((B, S, H, Dv), e["name"], "v"))
    do = to(testdata.normal_bf16((B, S, H, Dv), e["name"], "do"))
    out = torch.empty((B, S, H, Dv), dtype=torch.bfloat16, device=device)
    lse = torch.empty((2, B, H, S), dtype=torch.float32, device=device)
    desc = fa.make_desc(kind="diff", mask=e["mask"], diff_lambda=workloads.DIFF["lam"])
    fa.fl_attn_fwd(q, k, v, out, lse, desc)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fl_attn_diff_bwd_workspace_size(q, k, v, desc), dtype=torch.uint8, device=device)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            fa.fl_attn_diff_bwd(q, k, v, lse, do, dq, dk, dv, desc, ws, stream=stream)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fa.fl_attn_diff_bwd(q, k, v, lse, do, dq, dk, dv, desc, ws, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def decode_entry(mod):
    """The serving workload: one new token per sequence against a paged cache."""
    w = workloads.DECODE
    B, Sq, Hq, Hk, D = w["B"], w["Sq"], w["Hq"], w["Hk"], w["D"]
    lens = testdata.kv_lengths(B, w["name"], w["kv_lo"], w["kv_hi"]).astype(np.int64)
    keys = int(lens.sum())
    return dict(name=w["name"], kind="decode", variant="causal" if mod == "none" else "softcap",
                mod=mod, B=B, Sq=Sq, Hq=Hq, Hk=Hk, D=D, lens=lens, page=w["page"],
                flops=4 * D * Sq * Hq * keys,
                bytes=2 * 2 * keys * Hk * D + 2 * 2 * B * Sq * Hq * D + 4 * B * Hq * Sq)


def head_dim_entries():
    """The MHA S = 2048 shape at head dimensions 32 and 128."""
    return [entry("mha", 2048, v, D=D) for D in (32, 128) for v in ("vanilla", "causal")]


def all_entries():
    out = [entry("mha", S, v) for S in workloads.MHA_SEQ_LENS for v in workloads.MHA_VARIANTS]
    out += [entry("gqa", S, m) for S, _ in workloads.GQA_SHAPES for m in workloads.GQA_MASKS]
    return out


# ---------------------------------------------------------------- environment

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(bf16_tflops=d["bf16_tflops"], bf16_tflops_sustained=d["bf16_tflops_sustained"],
                    hbm_gbs=d["hbm_gbs"], source="measured")
    return dict(bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, hbm_gbs=6800.0,
                source="fallback")


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "std_fwd_mha_s2048_vanilla_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload)
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- ranks

def init_ranks():
    """(world, rank, local rank) from the torchrun environment; joins the
    process group when world > 1 (NCCL with a GPU, gloo otherwise)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def max_over_ranks(value, world, device):
    """The largest of every rank's value (the slowest rank's step time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, step_ms):
    """Whole-job rate: every rank's units over the slowest rank's time (per second)."""
    return units_per_rank * world / (step_ms * 1e-3)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"fl_bench_clocks_{os.getpid()}_{gpu_index}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, flag in zip(names, f[5:9]):
                if flag.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        busy = [x for x in sm if x >= 0.5 * (mx or 1)] or sm
        return dict(sm_mhz=statistics.median(busy), sm_max_mhz=mx, reasons=sorted(reasons),
                    samples=len(sm))


# ---------------------------------------------------------------- GPU arm

def gpu_inputs(e, torch, device):
    q = testdata.normal_bf16((e["B"], e["S"], e["Hq"], e["D"]), e["name"], "q")
    k = testdata.normal_bf16((e["B"], e["S"], e["Hk"], e["D"]), e["name"], "k")
    v = testdata.normal_bf16((e["B"], e["S"], e["Hk"], e["D"]), e["name"], "v")
    to = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    return [to(x) for x in (q, k, v)]


def time_entry(e, host, torch, fa, device, steps, warmup, flush, stream):
    q, k, v = (x.to(device) for x in host)
    out = torch.empty((e["B"], e["S"], e["Hq"], e["D"]), dtype=torch.bfloat16, device=device)
    lse = torch.empty((e["B"], e["Hq"], e["S"]), dtype=torch.float32, device=device)
    doc_t = torch.from_numpy(e["doc"]).to(device) if e["doc"] is not None else None
    desc = fa.make_desc(score_mod=e["mod"], mask=e["mask"], doc_offsets=doc_t,
                        softcap=workloads.SOFTCAP, **e["kw"])
    if e["mod"] == "expr":
        fa.fl_attn_fwd(q, k, v, out, lse, desc, stream=stream)  # the run-time compilation
        torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            fa.fl_attn_fwd(q, k, v, out, lse, desc, stream=stream)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for s, t in evs:
            flush.zero_()
            s.record(stream)
            fa.fl_attn_fwd(q, k, v, out, lse, desc, stream=stream)
            t.record(stream)
        torch.cuda.synchronize()
    ms = [s.elapsed_time(t) for s, t in evs]
    return ms, (q, k, v, out, lse, desc)


def time_other(e, torch, fa, device, steps, warmup, flush, stream):
    """Device time of the differential or Evoformer kernel on its workload."""
    to = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(device)
    if e["kind"] == "diff":
        B, S, H, D, Dv = e["B"], e["S"], e["H"], e["D"], e["Dv"]
        q = to(testdata.normal_bf16((2, B, S, H, D), e["name"], "q"))
        k = to(testdata.normal_bf16((2, B, S, H, D), e["name"], "k"))
        v = to(testdata.normal_bf16((B, S, H, Dv), e["name"], "v"))
        out = torch.empty((B, S, H, Dv), dtype=torch.bfloat16, device=device)
        lse = torch.empty((2, B, H, S), dtype=torch.float32, device=device)
        desc = fa.make_desc(kind="diff", mask=e["mask"], diff_lambda=workloads.DIFF["lam"])
        args = (q, k, v, out, lse, desc)
        kw = {}
    else:
        Ns, Nr, H, c = e["Ns"], e["Nr"], e["H"], e["c"]
        q, k, v, g = (to(testdata.normal_bf16((Ns, Nr, H, c), e["name"], n)) for n in "qkvg")
        out = torch.empty_like(q)
        row = e["kind"] == "evo_row"
        bias = to(testdata.normal_bf16((H, Nr, Nr), e["name"], "bias")) if row else None
        desc = fa.make_desc(kind=e["kind"])
        args = (q, k, v, out, None, desc)
        kw = dict(bias=bias, gate=g)
    flushed = l2_policy(e).startswith("flushed")
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            if flushed:
                flush.zero_()
            fa.fl_attn_fwd(*args, stream=stream, **kw)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            if flushed:
                flush.zero_()
            a.record(stream)
            fa.fl_attn_fwd(*args, stream=stream, **kw)
            b.record(stream)
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_evo_batched(e, torch, fa, device, steps, warmup, flush, stream):
    """Device time of fl_attn_evoformer over the batch of masked stacks (one
    launch per stack, all inside the timed region)."""
    to = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(device)
    shape = (e["Bt"], e["Ns"], e["Nr"], e["H"], e["c"])
    q, k, v, g = (to(testdata.normal_bf16(shape, e["name"], n)) for n in "qkvg")
    bias = to(testdata.normal_bf16((e["Bt"], e["H"], e["Nr"], e["Nr"]), e["name"], "bias")) \
        if e["row"] else None
    mask = torch.from_numpy(e["mask"]).to(device)
    out = torch.empty_like(q)
    desc = fa.make_desc(kind="evo_row" if e["row"] else "evo_col")
    flushed = l2_policy(e).startswith("flushed")
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            if flushed:
                flush.zero_()
            fa.fl_attn_evoformer(q, k, v, out, None, desc, bias=bias, gate=g, msa_mask=mask,
                                 stream=stream)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            if flushed:
                flush.zero_()
            a.record(stream)
            fa.fl_attn_evoformer(q, k, v, out, None, desc, bias=bias, gate=g, msa_mask=mask,
                                 stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_decode(e, torch, fa, device, steps, warmup, flush, stream):
    """Device time of the decode kernel on its workload (paged cache, pages of
    each sequence scattered over the pool)."""
    B, Sq, Hq, Hk, D, page = e["B"], e["Sq"], e["Hq"], e["Hk"], e["D"], e["page"]
    per = [-(-int(L) // page) for L in e["lens"]]
    n_pages = sum(per)
    perm = np.random.default_rng(7).permutation(n_pages).astype(np.int32)
    table = np.full((B, max(per)), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, : per[b]] = perm[at: at + per[b]]
        at += per[b]
    to = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
    q = to(testdata.normal_bf16((B, Sq, Hq, D), e["name"], "q"))
    kp = to(testdata.normal_bf16((n_pages, page, Hk, D), e["name"], "kpool"))
    vp = to(testdata.normal_bf16((n_pages, page, Hk, D), e["name"], "vpool"))
    out = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=device)
    lens_t = torch.from_numpy(e["lens"].astype(np.int32)).to(device)
    table_t = torch.from_numpy(table).to(device)
    d = fa.make_decode_desc(lens_t, int(e["lens"].max()), score_mod=e["mod"], softcap=workloads.SOFTCAP,
                            causal=True, block_table=table_t)
    ws = torch.empty(fa.fl_attn_decode_workspace_size(q, kp, d), dtype=torch.uint8, device=device)
    flushed = l2_policy(e).startswith("flushed")
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            if flushed:
                flush.zero_()
            fa.fl_attn_decode(q, kp, vp, out, lse, d, ws, stream=stream)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            if flushed:
                flush.zero_()
            a.record(stream)
            fa.fl_attn_decode(q, kp, vp, out, lse, d, ws, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_e2e(e, host, torch, fa, device, steps, warmup, stream):
    """Same metric end to end: every step copies its inputs from pinned host
    memory to the device, runs the fused forward and reads O and LSE back to
    pinned host memory.  Steps are pipelined over two device buffer sets and
    three streams (copy in, compute, copy out), so step n+1's upload overlaps
    step n's forward; the timed region runs from the first upload to the last
    download."""
    hq, hk, hv = (x.pin_memory() for x in host)
    sets = []
    for _ in range(2):
        q, k, v = (torch.empty_like(x, device=device) for x in host)
        out = torch.empty((e["B"], e["S"], e["Hq"], e["D"]), dtype=torch.bfloat16, device=device)
        lse = torch.empty((e["B"], e["Hq"], e["S"]), dtype=torch.float32, device=device)
        sets.append((q, k, v, out, lse))
    ho = torch.empty(sets[0][3].shape, dtype=torch.bfloat16).pin_memory()
    hl = torch.empty(sets[0][4].shape, dtype=torch.float32).pin_memory()
    desc = fa.make_desc(score_mod=e["mod"], mask=e["mask"], softcap=workloads.SOFTCAP, **e["kw"])
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_done = [ev(), ev()]
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    used = [False, False]

    def step(n):
        i = n & 1
        q, k, v, out, lse = sets[i]
        with torch.cuda.stream(s_in):
            if used[i]:
                s_in.wait_event(comp_done[i])   # step n-2's forward has read this set
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            in_done[i].record(s_in)
        stream.wait_event(in_done[i])
        if used[i]:
            stream.wait_event(out_done[i])      # step n-2's outputs have been read back
        fa.fl_attn_fwd(q, k, v, out, lse, desc, stream=stream)
        comp_done[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[i])
            ho.copy_(out, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
            out_done[i].record(s_out)
        used[i] = True

    for n in range(warmup):
        step(n)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for n in range(warmup, warmup + steps):
        step(n)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return ms, h2d, d2h, copy_rates(sets[0], (hq, hk, hv), (ho, hl), torch, s_in, s_out)


def copy_rates(dev_set, h_in, h_out, torch, s_in, s_out, reps=5):
    """The copies of one end-to-end step alone, each direction on its own
    stream with CUDA events (mean of `reps`): the pinned host-device link's
    rate for exactly these buffers, which bounds the pipelined step."""
    q, k, v, out, lse = dev_set

    def timed(stream, pairs):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for dst, src in pairs:      # warm the path once
                dst.copy_(src, non_blocking=True)
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(reps):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    up = timed(s_in, list(zip((q, k, v), h_in)))
    down = timed(s_out, list(zip(h_out, (out, lse))))
    nb_in = sum(x.numel() * x.element_size() for x in h_in)
    nb_out = sum(x.numel() * x.element_size() for x in h_out)
    return dict(h2d_ms=round(up, 4), d2h_ms=round(down, 4),
                h2d_gbs=round(nb_in / (up * 1e-3) / 1e9, 1), d2h_gbs=round(nb_out / (down * 1e-3) / 1e9, 1))


def cpu_baseline(e, seconds=12.0):
    """The oracle as it stands, on a bounded sample of query rows of the
    workload, on all host cores; returns TFLOP/s in the same algorithmic unit."""
    import oracle
    q, k, v = (testdata.normal_bf16((e["B"], e["S"], h, e["D"]), e["name"], n)
               for n, h in (("q", e["Hq"]), ("k", e["Hk"]), ("v", e["Hk"])))
    rng = np.random.default_rng(0)

    lo, hi = row_intervals(e["mask"], e["S"], e["kw"].get("window", 0), e["kw"].get("prefix", 0))

    def run(n):
        rows = np.stack([rng.integers(0, e["B"], n), rng.integers(0, e["Hq"], n),
                         rng.integers(0, e["S"], n)], axis=1)
        t0 = time.perf_counter()
        oracle.attention(q, k, v, mod=e["mod"], mask=e["mask"], softcap=workloads.SOFTCAP,
                         rows=rows, **e["kw"])
        dt = time.perf_counter() - t0
        pairs = int((hi[rows[:, 2]] - lo[rows[:, 2]]).sum())
        return dt, 4 * e["D"] * pairs, n

    dt, fl, n = run(2048)
    n2 = int(min(8_000_000, max(2048, 2048 * seconds / max(dt, 1e-4))))
    dt, fl, n = run(n2)
    return dict(value=fl / dt / 1e12, unit="TFLOP/s", cores=oracle.max_threads(), kind="oracle",
                sample=f"{n} random query rows (full key range each) of {e['name']} "
                       f"{e['variant']}, {dt:.1f} s")


ONLY = {"diff": lambda: diff_entry("none"), "diff_causal": lambda: diff_entry("causal"),
        "evo_row": lambda: evo_entry(True), "evo_col": lambda: evo_entry(False),
        "evo_c64_row": lambda: evo_entry(True, workloads.EVO_C64),
        "evo_c64_col": lambda: evo_entry(False, workloads.EVO_C64),
        "decode": lambda: decode_entry("none"), "decode_softcap": lambda: decode_entry("softcap"),
        "vanilla": lambda: entry("mha", 2048, "vanilla"), "causal": lambda: entry("mha", 2048, "causal"),
        "d128": lambda: entry("mha", 2048, "vanilla", D=128), "d32": lambda: entry("mha", 2048, "vanilla", D=32),
        "diff_dv64": lambda: diff_entry("none", Dv=64),
        "softcap": lambda: entry("mha", 2048, "softcap"), "alibi": lambda: entry("mha", 2048, "alibi"),
        "s512_vanilla": lambda: entry("mha", 512, "vanilla"), "s512_causal": lambda: entry("mha", 512, "causal"),
        "gqa16k_window": lambda: entry("gqa", 16384, "window"), "gqa16k_doc": lambda: entry("gqa", 16384, "doc"),
        "gqa16k_prefix": lambda: entry("gqa", 16384, "prefix"),
        "expr_softcap": lambda: expr_entry(2048, "expr_softcap"),
        "expr_alibi": lambda: expr_entry(2048, "expr_alibi"),
        "evo_af2_row": lambda: evo_batched_entry(True), "evo_af2_col": lambda: evo_batched_entry(False),
        "bwd": lambda: bwd_entry("none"), "bwd_causal": lambda: bwd_entry("causal"),
        "bwd_expr_softcap": lambda: bwd_entry("none", EXPR_VARIANTS["expr_softcap"][1]),
        "bwd_softcap": lambda: bwd_entry("none", mod="softcap"),
        "diff_bwd": lambda: diff_bwd_entry("none"), "diff_bwd_causal": lambda: diff_bwd_entry("causal")}


def run_only(args):
    """Time one workload alone (for profiling)."""
    import torch
    import attention_variant_gb300 as fa
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    fa.load_library()
    stream = torch.cuda.Stream(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    e = ONLY[args.only]()
    if e["kind"] in ("mha", "gqa"):
        ms = statistics.mean(time_entry(e, gpu_inputs(e, torch, device), torch, fa, device, args.steps,
                                        args.warmup, flush, stream)[0])
    else:
        timer = {"decode": time_decode, "evo_batched": time_evo_batched,
                 "bwd": time_bwd, "diff_bwd": time_diff_bwd}.get(e["kind"], time_other)
        ms = statistics.mean(timer(e, torch, fa, device, args.steps, args.warmup, flush, stream))
    print(json.dumps({"only": args.only, "ms": round(ms, 4),
                      "tflops": round(e["flops"] / (ms * 1e-3) / 1e12, 1),
                      "gbs": round(e["bytes"] / (ms * 1e-3) / 1e9, 1)}), flush=True)


def run_ours(args):
    import torch
    import attention_variant_gb300 as fa

    world, rank, local = init_ranks()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    fa.load_library()
    stream = torch.cuda.Stream(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    head = entry("mha", HEADLINE["S"], HEADLINE["variant"])
    host = gpu_inputs(head, torch, device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # headline, timed under the clock sampler (which also covers warm-up and a
    # short untimed run of the same kernel so that it collects several samples)
    barrier()
    with ClockSampler(local) as clk:
        time_entry(head, host, torch, fa, device, max(1, args.clock_steps), 0, flush, stream)
        t0 = time.perf_counter()
        ms, _ = time_entry(head, host, torch, fa, device, args.steps, args.warmup, flush, stream)
        barrier()
        wall = time.perf_counter() - t0
    clocks = clk.summary()
    step_ms = max_over_ranks(statistics.mean(ms), world, device)
    value = job_throughput(head["flops"], world, step_ms) / 1e12
    peaks = measured_peaks()
    achieved = head["flops"] / (statistics.mean(ms) * 1e-3) / 1e12

    e2e_ms, h2d, d2h, copies = time_e2e(head, host, torch, fa, device, max(3, args.steps),
                                        args.warmup, stream)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    # the pipelined step cannot beat its slowest stage: the upload, the
    # forward or the read-back (each on its own engine or stream)
    bound_ms = max(copies["h2d_ms"], copies["d2h_ms"], statistics.mean(ms))
    copies["ceiling_value"] = round(head["flops"] / (bound_ms * 1e-3) / 1e12, 1)
    e2e = dict(value=job_throughput(head["flops"], world, e2e_ms) / 1e12, unit="TFLOP/s",
               h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h, copy_ceiling=copies)

    variants = {}
    if not args.headline_only:
        for e in [diff_entry("none"), diff_entry("causal"), diff_entry("none", Dv=64), evo_entry(True),
                  evo_entry(False), evo_entry(True, workloads.EVO_C64), evo_entry(False, workloads.EVO_C64)]:
            vms = time_other(e, torch, fa, device, args.variant_steps, VARIANT_WARMUP, flush, stream)
            vm = statistics.mean(vms)
            if e["kind"].startswith("evo"):
                e["visited"] = e["pairs"]  # 128-key tiles: N_res 384 and N_seq 512 leave no partial tile
            tf = e["flops"] / (vm * 1e-3) / 1e12
            gbs = e["bytes"] / (vm * 1e-3) / 1e9
            rec = dict(tflops=round(tf, 1), frac_peak=round(tf / peaks["bf16_tflops"], 4),
                       ms=round(vm, 4), gbs=round(gbs, 1), **spread(vms), **bound_times(e, peaks))
            if e["kind"].startswith("evo"):
                rec["frac_hbm"] = round(gbs / peaks["hbm_gbs"], 4)
            rec["l2"] = l2_policy(e)
            variants[f"{e['name']}/{e['variant']}"] = rec
        for e in (evo_batched_entry(True), evo_batched_entry(False)):
            vms = time_evo_batched(e, torch, fa, device, args.variant_steps, VARIANT_WARMUP, flush, stream)
            vm = statistics.mean(vms)
            gbs = e["bytes"] / (vm * 1e-3) / 1e9
            variants[f"{e['name']}/{e['variant']}"] = dict(
                tflops=round(e["flops"] / (vm * 1e-3) / 1e12, 1), ms=round(vm, 4), gbs=round(gbs, 1),
                frac_hbm=round(gbs / peaks["hbm_gbs"], 4), **spread(vms), l2=l2_policy(e))
        for e in (bwd_entry("none"), bwd_entry("causal"), bwd_entry("none", mod="softcap"),
                  bwd_entry("none", EXPR_VARIANTS["expr_softcap"][1])):
            vms = time_bwd(e, torch, fa, device, args.variant_steps, VARIANT_WARMUP, flush, stream)
            vm = statistics.mean(vms)
            tf = e["flops"] / (vm * 1e-3) / 1e12
            variants[f"{e['name']}/{e['variant']}"] = dict(
                tflops=round(tf, 1), frac_peak=round(tf / peaks["bf16_tflops"], 4), ms=round(vm, 4),
                gbs=round(e["bytes"] / (vm * 1e-3) / 1e9, 1), **spread(vms), **bound_times(e, peaks),
                l2="flushed before every timed step (256 MiB write)")
        for e in (diff_bwd_entry("none"), diff_bwd_entry("causal")):
            vms = time_diff_bwd(e, torch, fa, device, args.variant_steps, VARIANT_WARMUP, flush, stream)
            vm = statistics.mean(vms)
            tf = e["flops"] / (vm * 1e-3) / 1e12
            variants[f"{e['name']}/{e['variant']}"] = dict(
                tflops=round(tf, 1), frac_peak=round(tf / peaks["bf16_tflops"], 4), ms=round(vm, 4),
                gbs=round(e["bytes"] / (vm * 1e-3) / 1e9, 1), **spread(vms), **bound_times(e, peaks),
                l2="flushed before every timed step (256 MiB write)")
        for e in (decode_entry("none"), decode_entry("softcap")):
            vms = time_decode(e, torch, fa, device, args.variant_steps, VARIANT_WARMUP, flush, stream)
            vm = statistics.mean(vms)
            gbs = e["bytes"] / (vm * 1e-3) / 1e9
            variants[f"{e['name']}/{e['variant']}"] = dict(
                tflops=round(e["flops"] / (vm * 1e-3) / 1e12, 1), ms=round(vm, 4), gbs=round(gbs, 1),
                frac_hbm=round(gbs / peaks["hbm_gbs"], 4), **spread(vms), **bound_times(e, peaks),
                l2=l2_policy(e))
        for e in all_entries() + [expr_entry(head["S"], n) for n in EXPR_VARIANTS] + head_dim_entries():
            h = host if e["name"] == head["name"] else gpu_inputs(e, torch, device)
            vms, _ = time_entry(e, h, torch, fa, device, args.variant_steps, VARIANT_WARMUP, flush, stream)
            vm = statistics.mean(vms)
            tf = e["flops"] / (vm * 1e-3) / 1e12
            bn = fa.fl_attn_tile_shape(fa.make_desc(), e["D"])[1]
            e["visited"] = visited_pairs(e["mask"], e["B"], e["Hq"], e["S"], bn, e["kw"].get("window", 0),
                                         e["kw"].get("prefix", 0), e["doc"])
            variants[f"{e['name']}/{e['variant']}"] = dict(
                tflops=round(tf, 1), frac_peak=round(tf / peaks["bf16_tflops"], 4),
                ms=round(vm, 4), gbs=round(e["bytes"] / (vm * 1e-3) / 1e9, 1), **spread(vms),
                visited_tflops=round(4 * e["D"] * e["visited"] / (vm * 1e-3) / 1e12, 1),
                **bound_times(e, peaks))

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": head["name"] + "/vanilla", "B": head["B"], "H": head["Hq"],
                   "S": head["S"], "D": head["D"], "variant": "vanilla non-causal",
                   "l2": "flushed before every timed step (256 MiB write)",
                   "parallelism": f"independent replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": recorded_traffic(head["name"] + "/vanilla"),
                     "peak_source": peaks["source"] + " bf16 burst"},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
        "variants": variants,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(head, seconds=args.cpu_seconds)
    # the figures the targets are stated in, last on the line so that a
    # truncated record still shows them
    tg = {"mha_s2048/vanilla frac of bf16 peak": line["roofline"]["frac"]}
    for key, field in (("evo_msa_s512_r384_h8_c32/row", "frac_hbm"),
                       ("evo_msa_s512_r384_h8_c32/col", "frac_hbm"),
                       ("diff_b4_s4096_h16/non-causal", "frac_peak"),
                       ("mha_s512/vanilla", "gbs"), ("mha_s2048/softcap", "frac_peak")):
        if key in variants:
            tg[f"{key} {field}"] = variants[key][field]
    line["targets"] = tg
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    head = entry("mha", HEADLINE["S"], HEADLINE["variant"])
    q, k, v = (testdata.normal_bf16((head["B"], head["S"], h, head["D"]), head["name"], n)
               for n, h in (("q", head["Hq"]), ("k", head["Hk"]), ("v", head["Hk"])))
    rng = np.random.default_rng(1)
    rows_per_step = 512

    def step():
        rows = np.stack([rng.integers(0, head["B"], rows_per_step),
                         rng.integers(0, head["Hq"], rows_per_step),
                         rng.integers(0, head["S"], rows_per_step)], axis=1)
        oracle.attention(q, k, v, rows=rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    flops = 4 * head["D"] * head["S"] * rows_per_step
    value = flops / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": head["name"] + "/vanilla", "B": head["B"], "H": head["Hq"],
                   "S": head["S"], "D": head["D"], "variant": "vanilla non-causal"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--variant-steps", type=int, default=5)
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", choices=sorted(ONLY), default=None,
                    help="time only this workload (profiling aid)")
    ap.add_argument("--clock-steps", type=int, default=3000,
                    help="untimed steps run under the clock sampler before the timed ones")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
