"""The synthetic workloads: shapes and variant lists, nothing computed.

They stand in for the pages' evaluation workloads (Flashlight talk notes,
"Evaluation: FlexAttention-supported variants": 16 heads, head dim 64,
sequence 512-16k at a constant 16k tokens, GQA 16/2; "Evaluation: complex
variants" and "End-to-end": differential attention, the AlphaFold Evoformer
MSA gated self-attention, and LLaMA-3.2-1B served by vLLM with causal and
softcap attention).  No dataset items are reproduced; every tensor is
drawn by :mod:`testdata`.
"""
from __future__ import annotations

TOKENS = 16384

# Small vanilla MHA problem the oracle finishes in well under a second.
SMALL_VANILLA = dict(name="mha_vanilla_b1_h2_s256_d64", B=1, H=2, S=256, D=64)

# MHA score_mod sweep: H=16, D=64, S in {512, 2048, 8192, 16384}, B = 16384/S.
MHA_SEQ_LENS = (512, 2048, 8192, 16384)
MHA_VARIANTS = ("vanilla", "alibi", "softcap", "causal")
MHA_HEADS = 16
HEAD_DIM = 64
SOFTCAP = 20.0

# GQA mask sweep: 16 query heads over 2 KV heads, D=64.
GQA_HQ, GQA_HK = 16, 2
GQA_SHAPES = ((16384, 1), (4096, 4))   # (S, B)
GQA_MASKS = ("window", "prefix", "doc")
WINDOW = 1024
PREFIX = 2048
DOC_LEN_RANGE = (256, 4096)

# Differential attention: B=4, S=4096, H=16, D_qk=64, D_v=128, lambda=0.8.
DIFF = dict(name="diff_b4_s4096_h16", B=4, S=4096, H=16, D=64, Dv=128, lam=0.8)

# Evoformer MSA gated self-attention: N_seq=512, N_res=384, H=8, c=32.
EVO = dict(name="evo_msa_s512_r384_h8_c32", N_seq=512, N_res=384, H=8, c=32)
# The pages' Evoformer kernel benchmark head shape (4 heads of dimension 64; the
# pages give no MSA size, so the c = 32 workload's MSA is used: same bytes).
EVO_C64 = dict(name="evo_msa_s512_r384_h4_c64", N_seq=512, N_res=384, H=4, c=64)
# A batch of AlphaFold2-sized MSA stacks (sequence length 256) with an MSA mask
# shaped like padding: the last 26 residues and the last 12 MSA rows removed.
EVO_AF2 = dict(name="evo_af2_b8_s128_r256_h8_c32", B=8, N_seq=128, N_res=256, H=8, c=32,
               pad_res=26, pad_seq=12)


def mha_workload(S: int) -> dict:
    return dict(name=f"mha_s{S}", B=TOKENS // S, H=MHA_HEADS, S=S, D=HEAD_DIM)


def gqa_workload(S: int, B: int) -> dict:
    return dict(name=f"gqa_s{S}_b{B}", B=B, Hq=GQA_HQ, Hk=GQA_HK, S=S, D=HEAD_DIM)


# Serving with a KV cache (decode): LLaMA-3.2-1B attention shapes -- 32 query
# heads over 8 KV heads, head dimension 64 -- one new token per sequence,
# 64 sequences whose cache lengths are uniform in [512, 8192] (a synthetic
# stand-in for a conversation trace; no trace item is reproduced), paged in
# 256-token pages.  Variants: causal (the new token sees its whole cache) and
# softcap (cap 20, as in the MHA sweep).
DECODE = dict(name="decode_llama1b_b64", B=64, Sq=1, Hq=32, Hk=8, D=64, kv_lo=512,
              kv_hi=8192, page=256, softcap=20.0)
