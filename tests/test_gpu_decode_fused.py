"""Decode as one cooperative launch (gather, K/V projection, gate, conv,
residual and state of every sequence) against the separate launches -- bit for
bit, the same arithmetic -- and against the oracle.

Cases vary the batch (one sequence; a partial 128-token row block; one
exactly; one and a half; the 256 sequences of the decode workload), take
several steps in a row from a streamed prefix, run without a state (fresh
sequences of one token), through engram_stage_b with the rows gathered
beforehand, and with int8 tables in HBM and in pinned host memory.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import engram_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from hashed_gram_embedding_engram_gb300 import EngramState  # noqa: E402
from tests.gpu_helpers import act_to_f64, assert_close, make_layer, to_torch  # noqa: E402

BASE = W.PREFILL_BF16.scaled(V=5000, V_proj=3850, prime_target=4001)
I8 = W.INT8_HOST.scaled(V=5000, V_proj=3850, prime_target=3001, span_copies=0, span_len=0)


def bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def run_steps(w, fused, prefix, steps, use_stage_b=False, table_on_host=False):
    """H and the state after a streamed prefix and `steps` one-token steps."""
    T = prefix + steps
    ids = W.token_stream(w.scaled(T=T))
    P = W.projection_map(w)
    L = W.layer_inputs(w.scaled(T=T), 1)
    plan, weights, proj, H = make_layer(w.scaled(T=T), L, P, w.B * T)
    if table_on_host:
        weights.table = to_torch(L.table, w.table_dtype, "cpu", pin=True)
    plan.set_fused_decode(fused)
    ids_d = torch.from_numpy(ids).cuda()
    st = EngramState.zeros(plan, w.B)
    if prefix:
        pre = H[:, :prefix].contiguous()
        plan.forward(ids_d[:, :prefix].contiguous(), proj, weights, pre, st)
        H[:, :prefix] = pre
    plan.set_timing(True)
    n_traced = None
    for t in range(prefix, T):
        step_ids = ids_d[:, t:t + 1].contiguous()
        step = H[:, t:t + 1].contiguous()
        if use_stage_b:
            e = plan.stage_a(step_ids, proj, weights.table, weights.scales, prev_ids=st.prev_ids)
            plan.stage_b(e, weights, step, st, ids=step_ids, proj=proj)
        else:
            plan.forward(step_ids, proj, weights, step, st)
        n_traced = len(plan.kernel_times())
        H[:, t:t + 1] = step
    plan.set_timing(False)
    assert plan.get_error() == (0, 0)
    return H, st, (ids, P, L, T), n_traced


@pytest.mark.parametrize("B", [1, 5, 128, 192, 256])
def test_fused_decode_equals_separate_launches(B):
    w = BASE.scaled(B=B, T=1)
    Hf, sf, _, nf = run_steps(w, True, 12, 3)
    Hs, ss, _, ns = run_steps(w, False, 12, 3)
    assert nf == 1 and ns == 3            # one traced interval for the fused step, three launches otherwise
    assert torch.equal(bits(Hf), bits(Hs))
    assert torch.equal(sf.prev_ids, ss.prev_ids) and torch.equal(sf.pos, ss.pos)
    assert torch.equal(bits(sf.u_ring), bits(ss.u_ring))


def test_fused_decode_matches_oracle_and_prefill():
    w = BASE.scaled(B=37, T=1)
    H, st, (ids, P, L, T), _ = run_steps(w, True, 9, 4)
    ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)
    assert_close(act_to_f64(H), ref["H_new"], "bf16", "fused decode")
    assert np.array_equal(st.prev_ids.cpu().numpy(), ref["state"]["prev"])
    assert torch.equal(st.pos.cpu(), torch.full((w.B,), T, dtype=torch.int32))
    # one-shot prefill of the same tokens gives the same bits
    plan, weights, proj, H0 = make_layer(w.scaled(T=T), L, P, w.B * T)
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H0)
    assert torch.equal(bits(H), bits(H0))


def test_fused_decode_without_state_and_through_stage_b():
    # fresh one-token sequences (no state): the window is pad + the token
    w = BASE.scaled(B=40, T=1)
    Hf, _, _, _ = run_steps(w, True, 0, 1)
    Hs, _, _, _ = run_steps(w, False, 0, 1)
    assert torch.equal(bits(Hf), bits(Hs))
    # Stage A gathered first, then engram_stage_b: the launch without its gather phase
    Hb, sb, _, nb = run_steps(w, True, 6, 2, use_stage_b=True)
    Hs, ss, _, _ = run_steps(w, False, 6, 2)
    assert nb == 1
    assert torch.equal(bits(Hb), bits(Hs)) and torch.equal(bits(sb.u_ring), bits(ss.u_ring))


@pytest.mark.parametrize("host", [False, True])
def test_fused_decode_int8_tables(host):
    w = I8.scaled(B=70, T=1, d=256)
    Hf, sf, _, _ = run_steps(w, True, 5, 2, table_on_host=host)
    Hs, ss, (ids, P, L, T), _ = run_steps(w, False, 5, 2, table_on_host=host)
    assert torch.equal(bits(Hf), bits(Hs)) and torch.equal(bits(sf.u_ring), bits(ss.u_ring))
    ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)
    assert_close(act_to_f64(Hf), ref["H_new"], "bf16", "fused int8 decode")
