"""Turn a seeded workload's numpy arrays into the library's torch-side objects.

Argument plumbing only (dtype views, host/device placement, the plan's
configuration fields): nothing here computes any part of the Engram layer.
Used by the GPU tests, ``bench.py`` and ``__graft_entry__.smoke()``; the oracle
never imports it.
"""
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
    """(plan, weights, projection map on the device, H on the device) of one layer."""
    plan = make_plan(w, L, max_tokens)
    weights = make_weights(w, L, table_on_host)
    proj = torch.from_numpy(P).cuda()
    H = to_torch(L.H, w.act_dtype)
    return plan, weights, proj, H
