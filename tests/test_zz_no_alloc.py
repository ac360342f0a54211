"""engram_forward_static_scratch: the forward for callers that cannot allocate.

Some callers (a host framework that owns the device allocator, a plugin host
that takes only plain calls, a latency-critical path where cudaMalloc is not
allowed) cannot give the library a workspace.  This entry point keeps its
scratch in a fixed device array inside the library.  Checked here through the
C ABI against engram_forward with a caller-provided workspace, on two calls in
a row (the array keeps the previous call's contents), and its size limit.
This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from hashed_gram_embedding_engram_gb300 import _lib  # noqa: E402
from tests.gpu_helpers import act_to_f64, make_layer, TOL  # noqa: E402

STATIC_SCRATCH_BYTES = 32 << 20


def call_static(plan, ids, proj, weights, H):
    w = weights.struct(plan)
    B, T = ids.shape
    return _lib._lib().engram_forward_static_scratch(
        plan._h, ids.data_ptr(), B, T, proj.data_ptr(), proj.numel(), ctypes.byref(w), H.data_ptr(), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_matches_forward_twice_in_a_row():
    w = W.PREFILL_BF16.scaled(B=3, T=333, V=5000, V_proj=3850, prime_target=4001, d=256)
    ids_np, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids_np.size)
    ids = torch.from_numpy(ids_np).cuda()
    assert plan.workspace_bytes(ids.numel()) <= STATIC_SCRATCH_BYTES

    ref = H0.clone()
    plan.forward(ids, proj, weights, ref)                  # caller-provided workspace
    tol_abs, tol_rel = TOL["bf16"]
    for _ in range(2):
        H = H0.clone()
        assert call_static(plan, ids, proj, weights, H) == _lib.OK
        torch.cuda.synchronize()
        got, exp = act_to_f64(H), act_to_f64(ref)
        diff = np.abs(got - exp)
        assert diff.max() <= tol_abs
        assert np.linalg.norm(got - exp) <= tol_rel * np.linalg.norm(exp)
    assert plan.get_error() == (0, 0)


def test_static_scratch_rejects_batches_beyond_its_size():
    w = W.PREFILL_BF16.scaled(B=1, T=8192, V=5000, V_proj=3850, prime_target=4001)
    ids_np, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids_np.size)
    assert plan.workspace_bytes(ids_np.size) > STATIC_SCRATCH_BYTES
    H0 = H.clone()
    st = call_static(plan, torch.from_numpy(ids_np).cuda(), proj, weights, H)
    assert st == _lib.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(H, H0)                              # nothing was launched
