"""Seeded synthetic inputs for the fused attention forward.

This module only draws numbers.  It holds none of the attention arithmetic, so
both the CPU oracle (``oracle/``) and the CUDA library's tests and benchmark can
take their inputs from it without sharing any code of the method.

Recipe (every tensor is reproducible from the global seed alone):

* sub-seed: ``splitmix64(GLOBAL_SEED ^ fnv1a64("<workload>/<tensor>/<index>"))``;
* stream: the n-th 64-bit draw is ``mix64(key + (n + 1) * GAMMA)`` -- the
  splitmix64 sequence started at ``key`` (Steele, Lea, Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014);
* normals: Box-Muller in double on consecutive draw pairs, using 53-bit
  uniforms in (0, 1); element 2m is the cosine branch, 2m+1 the sine branch;
* storage: double -> float32 (round to nearest) -> bfloat16 (round to nearest
  even).  The same bf16 bit patterns go to the GPU and to the oracle.
* document lengths: uniform integers in [256, 4096] drawn from the stream of
  ``"<workload>/doc_lengths/<batch>"`` until the running total reaches the
  sequence length; the last document is cut to fit.
* KV-cache lengths (serving workload): uniform integers in [lo, hi] drawn from
  the stream of ``"<workload>/kv_lengths/0"``, one per sequence.

The workloads themselves (shapes, variants) live in :mod:`testdata.workloads`.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GLOBAL_SEED = 20261202
GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1
_CHUNK = 1 << 20


def fnv1a64(text: str) -> int:
    """64-bit FNV-1a hash of a UTF-8 string."""
    h = 0xCBF29CE484222325
    for byte in text.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & _M64
    return h


def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(0xBF58476D1CE4E5B9)
        z ^= z >> np.uint64(27)
        z *= np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


def mix64_int(z: int) -> int:
    """Scalar splitmix64 output function."""
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def sub_seed(workload: str, tensor: str, index: int = 0, seed: int = GLOBAL_SEED) -> int:
    """Stream key of one tensor of one workload."""
    return mix64_int((seed ^ fnv1a64(f"{workload}/{tensor}/{index}")) + GAMMA)


def draws(key: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the splitmix64 stream at ``key``."""
    n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(key) + n * np.uint64(GAMMA)
    return mix64(state)


def _normal_chunk(key: int, first_pair: int, n_pairs: int) -> np.ndarray:
    d = draws(key, 2 * first_pair, 2 * n_pairs)
    u = ((d >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * n_pairs, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * math.pi * u2)
    out[1::2] = r * np.sin(2.0 * math.pi * u2)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, workload: str, tensor: str, index: int = 0,
                seed: int = GLOBAL_SEED, threads: int | None = None) -> np.ndarray:
    """N(0,1) samples of ``shape`` as bf16 bit patterns (uint16, C order)."""
    total = int(np.prod(shape))
    key = sub_seed(workload, tensor, index, seed)
    out = np.empty(total + (total & 1), dtype=np.uint16)
    pairs = (total + 1) // 2
    chunk_pairs = _CHUNK // 2

    def work(c0: int) -> None:
        n = min(chunk_pairs, pairs - c0)
        vals = _normal_chunk(key, c0, n).astype(np.float32)
        out[2 * c0: 2 * c0 + 2 * n] = f32_to_bf16_bits(vals)

    starts = list(range(0, pairs, chunk_pairs))
    if len(starts) == 1:
        work(0)
    else:
        nt = threads or min(len(starts), os.cpu_count() or 1)
        with ThreadPoolExecutor(max_workers=nt) as ex:
            list(ex.map(work, starts))
    return out[:total].reshape(shape)


def doc_lengths(seq_len: int, workload: str, batch_index: int,
                lo: int = 256, hi: int = 4096, seed: int = GLOBAL_SEED) -> list[int]:
    """Document lengths drawn uniformly from [lo, hi] until they cover ``seq_len``.

    The last document is truncated so the lengths sum to ``seq_len`` exactly.
    The integer is ``lo + draw % (hi - lo + 1)`` (modulo bias below 2^-52).
    """
    key = sub_seed(workload, "doc_lengths", batch_index, seed)
    lengths: list[int] = []
    total = 0
    n = 0
    while total < seq_len:
        d = int(draws(key, n, 1)[0])
        n += 1
        length = lo + d % (hi - lo + 1)
        length = min(length, seq_len - total)
        lengths.append(length)
        total += length
    return lengths


def kv_lengths(batch: int, workload: str, lo: int, hi: int, seed: int = GLOBAL_SEED) -> np.ndarray:
    """Per-sequence cache lengths, int32 ``[batch]``: ``lo + draw % (hi - lo + 1)``
    from the stream of ``"<workload>/kv_lengths/0"``."""
    key = sub_seed(workload, "kv_lengths", 0, seed)
    d = draws(key, 0, batch)
    return (lo + (d % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int32)


def doc_offsets(seq_len: int, batch: int, workload: str,
                lo: int = 256, hi: int = 4096, seed: int = GLOBAL_SEED) -> np.ndarray:
    """Document start offsets, int32 ``[batch, max_docs + 1]``.

    Row b holds the ascending starts of batch element b's documents (first is
    0) followed by ``seq_len`` repeated to fill the row.
    """
    rows = []
    for b in range(batch):
        lens = doc_lengths(seq_len, workload, b, lo, hi, seed)
        starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
        rows.append(starts)
    max_docs = max(len(r) for r in rows)
    table = np.full((batch, max_docs + 1), seq_len, dtype=np.int32)
    for b, r in enumerate(rows):
        table[b, : len(r)] = r
    return table
