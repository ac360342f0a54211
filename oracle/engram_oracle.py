"""Plain CPU oracle of the Engram conditional-memory forward path.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by ``bench.py``'s CPU-baseline / reference leg,
and by nothing else: the library never calls it, and it calls nothing of the
library.  It is deliberately slow and literal.

Source of every step: "DeepSeek Engram 系列导读" (foosynaptic.github.io,
deepseek-tech-notes, chapter 07-Engram), section "Engram 工作原理":
  Stage A (阶段 A：确定性检索)  Step 1 vocabulary projection, Step 2 suffix
  n-grams, Step 3 multi-head hashing, Step 4 concatenation;
  Stage B (阶段 B：上下文门控与融合)  Step 5 key/value projection, Step 6
  context-aware gate, Step 7 short dilated causal convolution, Step 8 residual;
  and the section "多分支 backbone 上的变体" for M hyper-connection branches.
The int8 row dequantisation follows "Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的
协同设计" (web.reeddaily.com), section "AgentX Engram DRAM卸载提升性能": one
kernel selects and dequantises rows, from HBM or pinned host memory; the page
gives no output precision, and the dequantised row is read as a bf16 row (it is
the input of the bf16 K/V projection).

Arithmetic: integers exactly (64-bit unsigned, wrap-around multiply); floating
point in float64, after exact widening of the stored inputs (fp32, bf16, and
int8 rows dequantised to bf16).  The pages fix no precision; apart from that
dequantised row nothing is rounded inside.

Readings where the pages leave a step open (each one is listed in the design
notes of the repository):
  * hash: h = XOR_{i<n} (x'_{t-i} * m_{n,k,i}) mod 2^64, z = h mod p_{n,k}
    (the page only says "multiplicative-XOR");
  * window slot i = 0 is x'_t itself (the n-gram is a suffix ending at t);
  * positions before the start of a sequence take projected id 0 (pad);
  * RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g, a separate weight g for h, for
    k and for the conv input; the gate scale sqrt(d) uses the hidden size d;
  * Conv1D is depthwise, causal, without bias, zero before the sequence start,
    PyTorch weight layout: tap j multiplies the input at lag (w-1-j)*dilation;
  * multi-branch: per-branch RMSNorm weights in the gate, shared W_V, conv
    weights and conv RMSNorm; branch m gets H^(m) += Y^(m);
  * FP8 projection (the section "多分支 backbone 上的变体" suggests one FP8 GEMM
    for [W_V; W_K^(1..M)] and says nothing more): e4m3 operands, one scale
    per row of e (per token) and per row of W_kv, s = amax/448, codes
    e4m3(x * (448/amax)) rounded to nearest even and saturated to +-448, the
    quotients and the product in binary32 (the codes are then a function of
    the stored inputs alone); the dot products of the codes are exact, the
    rest float64.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

MASK64 = np.uint64(0xFFFFFFFFFFFFFFFF)


# --------------------------------------------------------------------------- #
# stored formats -> exact float64
# --------------------------------------------------------------------------- #
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an IEEE binary32: widen the bit pattern exactly."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values that are exact in binary32 to bf16, nearest-even.

    Used only to state what a bf16 output of an exactly representable binary32
    value must be (int8 * fp16 products, which binary32 holds exactly)."""
    f32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), np.asarray(x, dtype=np.float64)), "not exact in binary32"
    u = f32.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def widen(x: np.ndarray, kind: str) -> np.ndarray:
    """Stored array -> float64: kind is 'f32' or 'bf16' (uint16 bit patterns)."""
    if kind == "bf16":
        return bf16_to_f64(x)
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------- #
# Stage A -- deterministic retrieval
# --------------------------------------------------------------------------- #
def project(ids: np.ndarray, P: np.ndarray) -> np.ndarray:
    """Step 1: x'_t = P(x_t), a precomputed many-to-one map of raw ids."""
    return np.asarray(P, dtype=np.int64)[np.asarray(ids, dtype=np.int64)]


def suffix_ngram(xp: np.ndarray, n: int, prev: Optional[np.ndarray] = None) -> List[np.ndarray]:
    """Step 2: g_{t,n} = (x'_{t-n+1}, ..., x'_t) for every t of every sequence.

    Returns [x'_{t-0}, x'_{t-1}, ..., x'_{t-n+1}], each [B, T].  ``prev`` holds
    the projected ids that precede position 0 of each sequence, oldest first
    ([B, >= n-1]); without it those positions are the pad id 0.  A window never
    reaches into another sequence of the batch."""
    B, T = xp.shape
    out = []
    for i in range(n):
        col = np.zeros((B, T), dtype=np.int64)
        col[:, i:] = xp[:, :T - i] if i < T else col[:, i:]
        if prev is not None and i > 0:
            for t in range(min(i, T)):
                # x'_{t-i} with t - i < 0 comes from prev, counted back from its end
                col[:, t] = prev[:, prev.shape[1] + (t - i)]
        out.append(col)
    return out


def multiplier(mults: np.ndarray, K: int, n: int, k: int, i: int) -> np.uint64:
    """m_{n,k,i}: the flat array is ordered n ascending, then k, then i."""
    base = sum(K * nn for nn in range(2, n))
    return np.uint64(mults[base + k * n + i])


def hash_heads(xp: np.ndarray, mults: np.ndarray, primes: Sequence[int], N: int, K: int,
               prev: Optional[np.ndarray] = None) -> np.ndarray:
    """Step 3: z_{t,n,k} = phi_{n,k}(g_{t,n}), K heads per order n = 2..N.

    phi_{n,k}(g) = (XOR_i x'_{t-i} * m_{n,k,i} mod 2^64) mod p_{n,k}.
    Returns int64 [B, T, (N-1)*K], head (n, k) in column (n-2)*K + k."""
    B, T = xp.shape
    z = np.empty((B, T, (N - 1) * K), dtype=np.int64)
    with np.errstate(over="ignore"):
        for n in range(2, N + 1):
            window = suffix_ngram(xp, n, prev)
            for k in range(K):
                h = np.zeros((B, T), dtype=np.uint64)
                for i in range(n):
                    h ^= window[i].astype(np.uint64) * multiplier(mults, K, n, k, i)
                p = np.uint64(primes[(n - 2) * K + k])
                z[:, :, (n - 2) * K + k] = (h % p).astype(np.int64)
    return z


def gather_concat(z: np.ndarray, tables: Sequence[np.ndarray], table_kind: str,
                  scales: Optional[Sequence[np.ndarray]] = None) -> np.ndarray:
    """Step 4: e_t = concat over n = 2..N, k = 1..K of E_{n,k}[z_{t,n,k}].

    table_kind: 'f32', 'bf16' (uint16 bits) or 'i8' (int8 rows, each times its
    fp16 row scale, dequantised to a bf16 row: the rows feed the bf16 K/V
    projection; the product is exact in binary32, so bf16(q*s) is one rounding).
    Returns float64 [..., R * row_dim]."""
    parts = []
    for r, E in enumerate(tables):
        rows = E[z[..., r]]
        if table_kind == "i8":
            s = np.asarray(scales[r], dtype=np.float16).astype(np.float64)[z[..., r]]
            parts.append(bf16_to_f64(f64_to_bf16_bits(rows.astype(np.float64) * s[..., None])))
        else:
            parts.append(widen(rows, table_kind))
    return np.concatenate(parts, axis=-1)


# --------------------------------------------------------------------------- #
# Stage B -- context-aware gating and fusion
# --------------------------------------------------------------------------- #
def kv_projection(e: np.ndarray, W_V: np.ndarray, W_K: Sequence[np.ndarray]):
    """Step 5: k_t = W_K e_t, v_t = W_V e_t (one W_K per branch)."""
    v = e @ W_V.T
    k = np.stack([e @ Wk.T for Wk in W_K], axis=-2)   # [..., M, d]
    return k, v


# --------------------------------------------------------------------------- #
# FP8 (e4m3) projection
# --------------------------------------------------------------------------- #
E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even), saturating to +-448.

    e4m3 (OCP 8-bit floating point, E4M3): sign, 4 exponent bits with bias 7,
    3 mantissa bits.  Normal values 2^(E-7) (1 + m/8), E = 1..15, except
    E = 15, m = 7 (NaN), so the largest finite value is 2^8 * 1.75 = 448;
    subnormals 2^-6 (m/8) = m * 2^-9.  On [2^k, 2^(k+1)) with k >= -6 the
    grid step is 2^(k-3); below 2^-6 it is 2^-9."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    step = np.where(a >= 2.0 ** -6, np.ldexp(1.0, ex - 1 - 3), 2.0 ** -9)
    q = np.minimum(np.round(a / step) * step, E4M3_MAX)    # np.round: half to even
    return np.copysign(q, x)


def quantize_rows_e4m3(x: np.ndarray):
    """Per-row e4m3 quantisation: (codes as float64 values, scales).

    s = amax/448 and q = e4m3(x * (448/amax)), both quotients and the product
    in binary32; an all-zero row gets s = 1 and zero codes."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1)).astype(np.float32)
    inv = np.where(nz, np.float32(E4M3_MAX) / safe, np.float32(0)).astype(np.float32)
    s = np.where(nz, safe / np.float32(E4M3_MAX), np.float32(1)).astype(np.float32)
    y = (x32 * inv[..., None]).astype(np.float32)
    return e4m3_round(y.astype(np.float64)), s.astype(np.float64)


def kv_projection_fp8(e: np.ndarray, W: np.ndarray, d: int, M: int):
    """Step 5 with e4m3 operands: kv = s_e s_w (q_e . q_w), then split into v and k^(1..M)."""
    qe, se = quantize_rows_e4m3(e)
    qw, sw = quantize_rows_e4m3(W)
    kv = (qe @ qw.T) * se[..., None] * sw
    v = kv[..., :d]
    k = np.stack([kv[..., (1 + m) * d:(2 + m) * d] for m in range(M)], axis=-2)
    return k, v


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps), times the weight g, over the last axis."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def gate(h: np.ndarray, k: np.ndarray, g_h: np.ndarray, g_k: np.ndarray, eps: float) -> np.ndarray:
    """Step 6: alpha_t = sigma(RMSNorm(h_t) . RMSNorm(k_t) / sqrt(d)); per branch.

    h, k: [..., M, d]; g_h, g_k: [M, d].  Returns alpha [..., M]."""
    d = h.shape[-1]
    dot = np.sum(rmsnorm(h, g_h, eps) * rmsnorm(k, g_k, eps), axis=-1)
    return sigmoid(dot / np.sqrt(d))


def dilated_causal_conv(u: np.ndarray, conv: np.ndarray, dil: int,
                        history: Optional[np.ndarray] = None) -> np.ndarray:
    """Depthwise causal Conv1D over the time axis of u [B, T, d].

    conv [d, w]: tap j multiplies u at lag (w-1-j)*dil.  Inputs before the
    first position are ``history`` (oldest first, [B, L, d]) or zero."""
    B, T, d = u.shape
    w = conv.shape[1]
    L = (w - 1) * dil
    if history is None:
        history = np.zeros((B, L, d))
    full = np.concatenate([history[:, history.shape[1] - L:], u], axis=1)   # index L + t is time t
    out = np.zeros_like(u)
    for j in range(w):
        lag = (w - 1 - j) * dil
        out += conv[:, j] * full[:, L - lag:L - lag + T]
    return out


def conv_branch(vt: np.ndarray, g_c: np.ndarray, conv: np.ndarray, dil: int, eps: float,
                vt_history: Optional[np.ndarray] = None) -> np.ndarray:
    """Step 7: Y = SiLU(Conv1D(RMSNorm(V~))) + V~ for one stream vt [B, T, d]."""
    u = rmsnorm(vt, g_c, eps)
    u_hist = None if vt_history is None else rmsnorm(vt_history, g_c, eps)
    c = dilated_causal_conv(u, conv, dil, u_hist)
    return c * sigmoid(c) + vt


# --------------------------------------------------------------------------- #
# the whole layer
# --------------------------------------------------------------------------- #
def forward(ids: np.ndarray, P: np.ndarray, L, N: int, K: int, dil: int, eps: float,
            table_kind: str, act_kind: str, state: Optional[Dict] = None,
            projection: str = "exact") -> Dict[str, np.ndarray]:
    """One Engram layer over a batch of sequences, Steps 1-8.

    ``L`` carries the layer's inputs (multipliers, primes, tables, scales, W_kv,
    g_h, g_k, g_c, conv, H as stored).  ``state`` continues sequences that
    already saw tokens: {'prev': [B, N-1] projected ids (oldest first),
    'vt_hist': [B, (w-1)*dil, M, d] float64 gated values (oldest first)}.
    Returns H_new (float64 [B,T,M,d]) with the intermediates and the state
    after the last position.  projection="fp8": Step 5 on e4m3 operands
    (kv_projection_fp8)."""
    B, T = ids.shape
    d = L.g_c.shape[0]
    M = L.g_h.shape[0]
    xp = project(ids, P)
    prev = None if state is None else state["prev"]
    z = hash_heads(xp, L.multipliers, L.primes, N, K, prev)
    e = gather_concat(z, L.tables(), table_kind, L.table_scales())
    W = widen(L.W_kv, act_kind)
    W_V = W[:d]
    W_K = [W[(1 + m) * d:(2 + m) * d] for m in range(M)]
    if projection == "fp8":
        k, v = kv_projection_fp8(e, W, d, M)
    else:
        k, v = kv_projection(e, W_V, W_K)                 # k [B,T,M,d], v [B,T,d]
    H = widen(L.H, act_kind)                              # [B,T,M,d]
    alpha = gate(H, k, L.g_h, L.g_k, eps)                 # [B,T,M]
    w = L.conv.shape[1]
    H_new = np.empty_like(H)
    vt_all = alpha[..., None] * v[:, :, None, :]          # [B,T,M,d]: branch m gets alpha^(m) * W_V e
    for m in range(M):
        hist = None if state is None else state["vt_hist"][:, :, m, :]
        Y = conv_branch(vt_all[:, :, m, :], L.g_c, L.conv, dil, eps, hist)
        H_new[:, :, m, :] = H[:, :, m, :] + Y             # Step 8
    # state after the last position
    Lh = (w - 1) * dil
    old_hist = np.zeros((B, Lh, M, d)) if state is None else state["vt_hist"]
    hist = np.concatenate([old_hist, vt_all], axis=1)[:, -Lh:]
    old_prev = np.zeros((B, N - 1), dtype=np.int64) if prev is None else prev
    new_prev = np.concatenate([old_prev, xp], axis=1)[:, -(N - 1):]
    return {"H_new": H_new, "z": z, "e": e, "k": k, "v": v, "alpha": alpha, "vt": vt_all,
            "state": {"prev": new_prev, "vt_hist": hist}}


def forward_at(ids: np.ndarray, P: np.ndarray, L, N: int, K: int, dil: int, eps: float,
               table_kind: str, act_kind: str, positions: Sequence, projection: str = "exact") -> np.ndarray:
    """Windowed re-evaluation: H_new at selected (b, t) from local inputs only.

    For each requested (b, t) this touches only the raw tokens x_{t'-i} of the
    positions t' = t - j*dil (j < w) that the convolution reads, and h at
    those t'.  It walks the definition position by position instead of
    shifting whole sequences, so it checks the full-sequence ``forward``'s
    windowing and padding.  Returns float64 [len(positions), M, d]."""
    d = L.g_c.shape[0]
    M = L.g_h.shape[0]
    w = L.conv.shape[1]
    W = widen(L.W_kv, act_kind)
    W_V = W[:d]
    W_K = [W[(1 + m) * d:(2 + m) * d] for m in range(M)]
    Pm = np.asarray(P, dtype=np.int64)
    tabs, scs = L.tables(), L.table_scales()

    # every position t' whose gated value some requested output needs
    need = sorted({(b, t - j * dil) for (b, t) in positions for j in range(w) if t - j * dil >= 0})
    slot = {bt: i for i, bt in enumerate(need)}
    zrows = np.empty((len(need), (N - 1) * K), dtype=np.int64)
    with np.errstate(over="ignore"):
        for i, (b, tp) in enumerate(need):
            for n in range(2, N + 1):
                for k in range(K):
                    h = np.uint64(0)
                    for s in range(n):
                        x = Pm[ids[b, tp - s]] if tp - s >= 0 else 0
                        h ^= np.uint64(x) * multiplier(L.multipliers, K, n, k, s)
                    zrows[i, (n - 2) * K + k] = int(h % np.uint64(L.primes[(n - 2) * K + k]))
    e = gather_concat(zrows, tabs, table_kind, scs)                    # [n_need, d_mem]
    if projection == "fp8":
        k, v = kv_projection_fp8(e, W, d, M)
    else:
        k, v = kv_projection(e, W_V, W_K)                              # [n_need, M, d], [n_need, d]
    Hn = np.stack([widen(L.H[b, tp], act_kind) for (b, tp) in need])   # [n_need, M, d]
    alpha = gate(Hn, k, L.g_h, L.g_k, eps)                             # [n_need, M]
    vt = alpha[..., None] * v[:, None, :]                              # [n_need, M, d]
    u = rmsnorm(vt, L.g_c, eps)

    out = np.empty((len(positions), M, d))
    for o, (b, t) in enumerate(positions):
        c = np.zeros((M, d))
        for j in range(w):
            tp = t - (w - 1 - j) * dil
            if tp >= 0:
                c += L.conv[:, j] * u[slot[(b, tp)]]
        Y = c * sigmoid(c) + vt[slot[(b, t)]]
        out[o] = widen(L.H[b, t], act_kind) + Y
    return out
