"""Glue between the seeded workloads (numpy) and the library's torch front end."""
from __future__ import annotations

import numpy as np
import torch

from workloads.torch_layer import make_layer, make_plan, make_weights, to_torch  # noqa: F401


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


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

    For bf16 the max-abs bound is 2e-2 except where |ref| >= 8: there the
    spacing of bf16 numbers is 0.0625, so no bf16 value lies within 2e-2 of
    every real.  A stored output is the fp32 result (within 2e-2 of the real
    one) rounded once to bf16, which moves it by at most half a bf16 ulp at
    its own magnitude (at most |ref| + 2e-2), so the bound there is
    2e-2 + ulp/2 (0.05125 on [8, 16 - 2e-2)).  The relative-L2 bound applies
    unchanged."""
    tol_abs, tol_rel = TOL[kind]
    mx, rel = errors(got, ref)
    diff = np.abs(got - ref)
    bound = np.where(np.abs(ref) < 8, tol_abs, tol_abs + 0.5 * bf16_ulp(np.abs(ref) + tol_abs)) if kind == "bf16" else tol_abs
    worst = float((diff - bound).max())
    assert worst <= 0.0 and rel <= tol_rel, f"{what}: max-abs {mx:.4g}, rel-L2 {rel:.4g}, worst excess {worst:.3g}"
