"""Glue between the seeded workloads (numpy) and the library's torch front end."""
from __future__ import annotations

import numpy as np
import torch

from hashed_gram_embedding_engram_gb300 import EngramPlan, EngramWeights


def to_torch(a: np.ndarray, kind: str, device="cuda", pin: bool = False) -> torch.Tensor:
    """numpy array as stored by the generators -> torch tensor of the stored dtype."""
    if kind == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    if device == "cpu":
        return t.pin_memory() if pin else t
    return t.to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_plan(w, L, max_tokens: int) -> EngramPlan:
    return EngramPlan(N=w.N, K=w.K, row_dim=w.row_dim, d=w.d, M=w.M, conv_w=w.conv_w, conv_dilation=w.conv_dil,
                      table_dtype=w.table_dtype, act_dtype=w.act_dtype, eps=w.eps, primes=L.primes.tolist(),
                      multipliers=[int(m) for m in L.multipliers], max_tokens=max_tokens)


def make_weights(w, L, table_on_host: bool = False) -> EngramWeights:
    dev = "cpu" if table_on_host else "cuda"
    table = to_torch(L.table, w.table_dtype, dev, pin=table_on_host)
    scales = None
    if L.scales is not None:
        scales = to_torch(L.scales, "f16", "cuda")
    return EngramWeights(table=table, w_kv=to_torch(L.W_kv, w.act_dtype), g_h=to_torch(L.g_h, "f32"),
                         g_k=to_torch(L.g_k, "f32"), g_c=to_torch(L.g_c, "f32"), conv=to_torch(L.conv, "f32"),
                         scales=scales)


def make_layer(w, L, P, max_tokens: int, table_on_host: bool = False):
    plan = make_plan(w, L, max_tokens)
    weights = make_weights(w, L, table_on_host)
    proj = torch.from_numpy(P).cuda()
    H = to_torch(L.H, w.act_dtype)
    return plan, weights, proj, H


def act_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    diff = got - ref
    return float(np.abs(diff).max()), float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))


# Tolerances.  bf16 outputs: max-abs 2e-2 and relative L2 5e-3 against the
# float64 oracle.  fp32 outputs: derived from binary32 rounding (unit round-off
# 6e-8) over d_mem-long dot products and O(1) values: max-abs 1e-4, rel-L2 1e-5.
TOL = {"bf16": (2e-2, 5e-3), "f32": (1e-4, 1e-5)}


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def assert_close(got: np.ndarray, ref: np.ndarray, kind: str, what: str = "") -> None:
    """got (as stored: bf16 or fp32, widened) vs the float64 oracle.

    For bf16 the max-abs bound is 2e-2 except where |ref| >= 8: there one bf16
    ulp is 0.0625 and no bf16 value lies within 2e-2 of every real, so the bound
    there is one bf16 ulp.  The relative-L2 bound applies unchanged."""
    tol_abs, tol_rel = TOL[kind]
    mx, rel = errors(got, ref)
    diff = np.abs(got - ref)
    bound = np.where(np.abs(ref) < 8, tol_abs, bf16_ulp(ref)) if kind == "bf16" else tol_abs
    worst = float((diff - bound).max())
    assert worst <= 0.0 and rel <= tol_rel, f"{what}: max-abs {mx:.4g}, rel-L2 {rel:.4g}, worst excess {worst:.3g}"
