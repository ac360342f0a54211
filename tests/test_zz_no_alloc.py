"""engram_forward_static_scratch: the forward for callers that cannot allocate.

Some callers cannot give the library a workspace: code inside a host framework
that owns the device allocator and exposes none of it, a plugin host that takes
only plain calls, a latency-critical path where cudaMalloc (which may
synchronise the device) is not allowed.  This entry point keeps its scratch in
a fixed device array inside the library.

Checked here through the C ABI: on two calls in a row (the array keeps the
previous call's contents) its output equals engram_forward's with a
caller-provided workspace bit for bit -- the same kernels on the same inputs --
for the two-launch prefill path, for Stage B as one cooperative launch (whose
counters live in the scratch and must be re-zeroed by every call) and for
decode steps with a streaming state; the device's free memory does not change
across the calls; batches beyond the array are refused before any launch.
This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from hashed_gram_embedding_engram_gb300 import EngramState, _lib  # noqa: E402
from tests.gpu_helpers import make_layer  # noqa: E402

STATIC_SCRATCH_BYTES = 32 << 20


def call_static(plan, ids, proj, weights, H, state=None):
    w = weights.struct(plan)
    B, T = ids.shape
    st = None if state is None else ctypes.byref(state.struct(plan, B))
    return _lib._lib().engram_forward_static_scratch(
        plan._h, ids.data_ptr(), B, T, proj.data_ptr(), proj.numel(), ctypes.byref(w), H.data_ptr(), st,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def layer(w):
    ids_np, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids_np.size)
    return plan, weights, proj, H0, torch.from_numpy(ids_np).cuda()


@pytest.mark.parametrize("fused_stage_b", [False, True])
def test_static_scratch_matches_forward_twice_in_a_row(fused_stage_b):
    # d = 1024, one branch, T > 1: the prefill path's kernel instances, and the
    # shape on which Stage B can run as one cooperative launch
    w = W.PREFILL_BF16.scaled(B=2, T=1000, V=5000, V_proj=3850, prime_target=4001)
    plan, weights, proj, H0, ids = layer(w)
    assert plan.workspace_bytes(ids.numel()) <= STATIC_SCRATCH_BYTES
    plan.set_fused_stage_b(fused_stage_b)

    ref = H0.clone()
    plan.forward(ids, proj, weights, ref)                  # caller-provided workspace
    H = H0.clone()
    assert call_static(plan, ids, proj, weights, H) == _lib.OK   # first call on the device: set-up
    assert bits_equal(H, ref)
    free0 = free_bytes()
    for _ in range(2):
        H.copy_(H0)
        assert call_static(plan, ids, proj, weights, H) == _lib.OK
        torch.cuda.synchronize()
        assert bits_equal(H, ref)
    assert free_bytes() == free0                           # nothing allocated on the device
    assert plan.get_error() == (0, 0)


def test_static_scratch_decode_steps_with_state():
    # 48 sequences: a 20-token prefix (plain forward), then two one-token steps
    # through both entry points from identical states
    w = W.PREFILL_BF16.scaled(B=48, T=22, V=5000, V_proj=3850, prime_target=4001, d=256)
    plan, weights, proj, H0, ids = layer(w)
    st = EngramState.zeros(plan, w.B)
    plan.forward(ids[:, :20].contiguous(), proj, weights, H0[:, :20].contiguous(), st)
    st_ref, st_got = st.clone(), st.clone()
    for t in (20, 21):
        step_ids = ids[:, t:t + 1].contiguous()
        ref = H0[:, t:t + 1].contiguous()
        got = ref.clone()
        plan.forward(step_ids, proj, weights, ref, st_ref)
        assert call_static(plan, step_ids, proj, weights, got, st_got) == _lib.OK
        torch.cuda.synchronize()
        assert bits_equal(got, ref)
        assert torch.equal(st_got.prev_ids, st_ref.prev_ids) and torch.equal(st_got.pos, st_ref.pos)
        assert torch.equal(st_got.u_ring.view(torch.int32), st_ref.u_ring.view(torch.int32))
    assert plan.get_error() == (0, 0)


def test_static_scratch_rejects_batches_beyond_its_size():
    w = W.PREFILL_BF16.scaled(B=1, T=8192, V=5000, V_proj=3850, prime_target=4001)
    plan, weights, proj, H, ids = layer(w)
    assert plan.workspace_bytes(ids.numel()) > STATIC_SCRATCH_BYTES
    H0 = H.clone()
    st = call_static(plan, ids, proj, weights, H)
    assert st == _lib.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(H, H0)                              # nothing was launched
