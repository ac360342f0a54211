"""Seeded synthetic inputs for the Engram layer.

This module only draws numbers; it holds none of the layer's arithmetic.  Both
the CPU oracle and the CUDA path receive exactly the arrays built here.

Recipe (all seeded from ``Workload.base_seed`` / ``weight_seed``):

* token ids: bounded Zipf, Pr(rank r) ~ r^-s for r = 1..V, drawn by inverse CDF,
  raw id = sigma(r-1) for a seeded permutation sigma of [0, V).  Per sequence one
  motif of ``span_len`` tokens (same Zipf) is pasted into ``span_copies`` distinct
  aligned slots, so the motif's n-grams repeat.
* projection P: V -> V': a seeded permutation pi of [0, V); P[pi[i]] = i for the
  first V' entries (so P is onto [0, V')), uniform seeded targets for the rest.
* hash multipliers: splitmix64 (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014) started from ``seed + layer_id``,
  drawn for order n ascending, head k ascending, window slot i ascending, each
  forced odd.  Seed 1 for the tiny workload, 20260112 for the others.
* primes: the first R primes >= ``prime_target``, assigned to (n, k) n-major.
* tables: N(0, table_std) rows, stored fp32, bf16 (round-to-nearest-even of an
  fp32 draw), or int8 with an fp16 per-row scale s = fp16(max|x| / 127),
  q = clamp(rint(x / s), -127, 127) (s = 1 for an all-zero row).
* H ~ N(0, h_std); W_V, W_K ~ N(0, w_std or 1/sqrt(d_mem)); RMSNorm weights
  1 + N(0, norm_std); depthwise conv weights N(0, conv_std).

Large arrays are filled in fixed-size chunks, each chunk with its own
``SeedSequence`` child, on a thread pool: the result does not depend on the
number of threads.
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import List, Optional

import numpy as np

from .configs import Workload

MASK64 = (1 << 64) - 1
_CHUNK = 1 << 24  # elements per independently seeded chunk


# --------------------------------------------------------------------------- #
# elementary generators
# --------------------------------------------------------------------------- #
def splitmix64(state: int, count: int) -> List[int]:
    """``count`` outputs of splitmix64 starting from ``state`` (Python ints)."""
    out = []
    s = state & MASK64
    for _ in range(count):
        s = (s + 0x9E3779B97F4A7C15) & MASK64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        out.append(z ^ (z >> 31))
    return out


def first_primes_from(target: int, count: int) -> List[int]:
    """The first ``count`` primes >= ``target`` (trial division)."""
    def isprime(n: int) -> bool:
        if n < 2:
            return False
        if n % 2 == 0:
            return n == 2
        f = 3
        while f * f <= n:
            if n % f == 0:
                return False
            f += 2
        return True

    out, n = [], target
    while len(out) < count:
        if isprime(n):
            out.append(n)
        n += 1
    return out


def _rng(seed: int, *key) -> np.random.Generator:
    words = []
    for k in key:
        words.append(zlib.crc32(k.encode()) if isinstance(k, str) else int(k))
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(words))))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _chunked_fill(n: int, fn, *key_seed) -> None:
    """Call fn(rng, lo, hi) for each chunk of [0, n), in parallel."""
    seed, key = key_seed[0], key_seed[1:]
    chunks = [(c, c * _CHUNK, min(n, (c + 1) * _CHUNK)) for c in range((n + _CHUNK - 1) // _CHUNK)]

    def run(item):
        c, lo, hi = item
        fn(_rng(seed, *key, c), lo, hi)

    if len(chunks) <= 1:
        for it in chunks:
            run(it)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(run, chunks))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns.

    Data preparation only (the inputs contain no NaN)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def normal_array(shape, std: float, dtype: str, seed: int, *key) -> np.ndarray:
    """N(0, std) array of ``shape`` stored as float32 or bf16 bits (uint16)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)

    def fill(rng, lo, hi):
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        x *= np.float32(std)
        out[lo:hi] = x if dtype == "f32" else f32_to_bf16_bits(x)

    _chunked_fill(n, fill, seed, *key)
    return out.reshape(shape)


def int8_rowscale_table(rows: int, row_dim: int, std: float, seed: int, *key):
    """int8 rows + fp16 per-row scales of an N(0, std) table (symmetric, per row)."""
    q = np.empty((rows, row_dim), dtype=np.int8)
    s = np.empty(rows, dtype=np.float16)
    rows_per_chunk = max(1, _CHUNK // row_dim)
    n = rows * row_dim

    def fill(rng, lo, hi):
        r0, r1 = lo // row_dim, hi // row_dim
        x = rng.standard_normal((r1 - r0, row_dim), dtype=np.float32)
        x *= np.float32(std)
        amax = np.abs(x).max(axis=1)
        sc = (amax / np.float32(127.0)).astype(np.float16)
        sc[amax == 0] = np.float16(1.0)
        qq = np.rint(x / sc.astype(np.float32)[:, None])
        q[r0:r1] = np.clip(qq, -127, 127).astype(np.int8)
        s[r0:r1] = sc

    assert _CHUNK % row_dim == 0 and rows_per_chunk * row_dim == _CHUNK
    _chunked_fill(n, fill, seed, *key)
    return q, s


def bounded_zipf(rng: np.random.Generator, V: int, s: float, size, sigma: np.ndarray) -> np.ndarray:
    """Raw ids: rank r ~ r^-s on 1..V by inverse CDF, mapped through sigma."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    u = rng.random(size)
    r = np.searchsorted(cdf, u, side="right")
    r = np.minimum(r, V - 1)
    return sigma[r].astype(np.int32)


# --------------------------------------------------------------------------- #
# per-workload inputs
# --------------------------------------------------------------------------- #
def token_stream(w: Workload, B: Optional[int] = None, T: Optional[int] = None, key: str = "tokens") -> np.ndarray:
    """int32 [B, T] raw token ids with repeated spans."""
    B = w.B if B is None else B
    T = w.T if T is None else T
    rng = _rng(w.base_seed, key)
    sigma = _rng(w.base_seed, "zipf-permutation").permutation(w.V)
    ids = bounded_zipf(rng, w.V, w.zipf_s, (B, T), sigma)
    if w.span_len and w.span_copies and T >= w.span_len:
        slots = T // w.span_len
        for b in range(B):
            motif = bounded_zipf(rng, w.V, w.zipf_s, w.span_len, sigma)
            n = min(w.span_copies, slots)
            chosen = rng.choice(slots, size=n, replace=False)
            for c in chosen:
                ids[b, c * w.span_len:(c + 1) * w.span_len] = motif
    return ids


def projection_map(w: Workload) -> np.ndarray:
    """int32 [V]: many-to-one onto [0, V')."""
    rng = _rng(w.weight_seed, "projection")
    pi = rng.permutation(w.V)
    P = np.empty(w.V, dtype=np.int32)
    P[pi[:w.V_proj]] = np.arange(w.V_proj, dtype=np.int32)
    P[pi[w.V_proj:]] = rng.integers(0, w.V_proj, size=w.V - w.V_proj, dtype=np.int32)
    return P


def hash_multipliers(w: Workload, layer_id: int) -> np.ndarray:
    """uint64 [sum_n K*n]: flat index of (n, k, i) is sum_{n'<n} K*n' + k*n + i."""
    seed = 1 if w.name.startswith("tiny") else 20260112
    vals = splitmix64(seed + layer_id, w.multiplier_count)
    return np.array([v | 1 for v in vals], dtype=np.uint64)


@dataclass
class LayerInputs:
    layer_id: int
    multipliers: np.ndarray   # uint64 [sum_n K*n]
    primes: np.ndarray        # uint32 [R], (n, k) n-major
    row_offsets: np.ndarray   # int64 [R], first row of table r in ``table``
    table: np.ndarray         # [sum p, row_dim]: float32 | uint16 (bf16 bits) | int8
    scales: Optional[np.ndarray]  # float16 [sum p] for int8 tables
    W_kv: np.ndarray          # [(M+1)d, d_mem]: rows [0,d) = W_V, [(1+m)d,(2+m)d) = W_K^(m)
    g_h: np.ndarray           # float32 [M, d] RMSNorm weight on h (per branch)
    g_k: np.ndarray           # float32 [M, d] RMSNorm weight on k (per branch)
    g_c: np.ndarray           # float32 [d]    RMSNorm weight before the conv
    conv: np.ndarray          # float32 [d, w] depthwise taps, tap w-1 = lag 0
    H: np.ndarray             # [B, T, M, d]: float32 | uint16 (bf16 bits)

    def tables(self) -> List[np.ndarray]:
        """Per-(n,k) views E_{n,k} of the concatenated table, n-major."""
        return [self.table[o:o + int(p)] for o, p in zip(self.row_offsets, self.primes)]

    def table_scales(self) -> Optional[List[np.ndarray]]:
        if self.scales is None:
            return None
        return [self.scales[o:o + int(p)] for o, p in zip(self.row_offsets, self.primes)]

    def W_V(self) -> np.ndarray:
        d = self.g_c.shape[0]
        return self.W_kv[:d]

    def W_K(self, m: int) -> np.ndarray:
        d = self.g_c.shape[0]
        return self.W_kv[(1 + m) * d:(2 + m) * d]


def layer_inputs(w: Workload, layer_id: int, B: Optional[int] = None, T: Optional[int] = None,
                 h_key: str = "H") -> LayerInputs:
    B = w.B if B is None else B
    T = w.T if T is None else T
    ws = w.weight_seed
    primes = np.array(first_primes_from(w.prime_target, w.R), dtype=np.uint32)
    offsets = np.zeros(w.R, dtype=np.int64)
    offsets[1:] = np.cumsum(primes.astype(np.int64))[:-1]
    rows = int(primes.astype(np.int64).sum())
    scales = None
    if w.table_dtype == "i8":
        table, scales = int8_rowscale_table(rows, w.row_dim, w.table_std, ws, layer_id, "table")
    else:
        table = normal_array((rows, w.row_dim), w.table_std, w.table_dtype, ws, layer_id, "table")
    w_std = w.w_std if w.w_std else 1.0 / np.sqrt(w.d_mem)
    W_kv = normal_array(((w.M + 1) * w.d, w.d_mem), w_std, w.act_dtype, ws, layer_id, "W_kv")
    rng = _rng(ws, layer_id, "norms")
    g_h = (1.0 + w.norm_std * rng.standard_normal((w.M, w.d))).astype(np.float32)
    g_k = (1.0 + w.norm_std * rng.standard_normal((w.M, w.d))).astype(np.float32)
    g_c = (1.0 + w.norm_std * rng.standard_normal(w.d)).astype(np.float32)
    conv = (w.conv_std * _rng(ws, layer_id, "conv").standard_normal((w.d, w.conv_w))).astype(np.float32)
    H = normal_array((B, T, w.M, w.d), w.h_std, w.act_dtype, w.base_seed, layer_id, h_key)
    return LayerInputs(layer_id, hash_multipliers(w, layer_id), primes, offsets, table, scales,
                       W_kv, g_h, g_k, g_c, conv, H)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for test and bench helpers)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
