"""Checkpoint and resume of the streaming (decode) state.

The state of B sequences -- the last N-1 projected ids, the conv ring of the
last (w-1)*dilation normalised inputs and the position -- is saved after step
s (serialised to bytes on the host), loaded into fresh device tensors, and
step s+1 from the loaded state must equal step s+1 of the uninterrupted run
bit for bit, in H and in the state it leaves.
"""
import io

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from hashed_gram_embedding_engram_gb300 import EngramState  # noqa: E402
from tests.gpu_helpers import make_layer  # noqa: E402


def save(st: EngramState) -> bytes:
    buf = io.BytesIO()
    torch.save({"prev_ids": st.prev_ids.cpu(), "u_ring": st.u_ring.cpu(), "pos": st.pos.cpu()}, buf)
    return buf.getvalue()


def load(blob: bytes) -> EngramState:
    d = torch.load(io.BytesIO(blob))
    return EngramState(d["prev_ids"].cuda(), d["u_ring"].cuda(), d["pos"].cuda())


@pytest.mark.parametrize("fused", [False, True])
def test_decode_state_checkpoint_resume_is_bit_identical(fused):
    w = W.PREFILL_BF16.scaled(B=24, T=1, V=5000, V_proj=3850, prime_target=4001, d=256)
    steps = 7
    T = 10 + steps
    ids = torch.from_numpy(W.token_stream(w.scaled(T=T))).cuda()
    P = W.projection_map(w)
    L = W.layer_inputs(w.scaled(T=T), 1)
    plan, weights, proj, H = make_layer(w.scaled(T=T), L, P, w.B * T)
    plan.set_fused_decode(fused)
    st = EngramState.zeros(plan, w.B)
    pre = H[:, :10].contiguous()
    plan.forward(ids[:, :10].contiguous(), proj, weights, pre, st)
    s = 10 + 3
    for t in range(10, s):                    # steps before the checkpoint
        h = H[:, t:t + 1].contiguous()
        plan.forward(ids[:, t:t + 1].contiguous(), proj, weights, h, st)
    torch.cuda.synchronize()
    blob = save(st)
    resumed = load(blob)
    for t in range(s, T):                     # both runs continue from the same point
        h_run = H[:, t:t + 1].contiguous()
        h_res = h_run.clone()
        plan.forward(ids[:, t:t + 1].contiguous(), proj, weights, h_run, st)
        plan.forward(ids[:, t:t + 1].contiguous(), proj, weights, h_res, resumed)
        assert torch.equal(h_run.view(torch.int16), h_res.view(torch.int16)), t
    assert torch.equal(st.prev_ids, resumed.prev_ids) and torch.equal(st.pos, resumed.pos)
    assert torch.equal(st.u_ring.view(torch.int32), resumed.u_ring.view(torch.int32))
    assert plan.get_error() == (0, 0)
