"""The five workloads at their full sizes, on the GPU, against the CPU oracle.

Integer work (indices, gathered rows) is compared in full, bit for bit.  The
layer output is compared in full where the float64 oracle finishes in seconds
(tiny, prefill, decode) and on sampled positions otherwise (int8 host tables,
multi-branch), using the oracle's windowed evaluator; the sample always holds
the first positions of every sequence and the last one.
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
from tests.gpu_helpers import act_to_f64, assert_close, bf16_bits, make_layer, to_torch  # noqa: E402

CHUNK = 8192   # tokens per comparison block (bounds host memory of the float64 oracle)


def check_indices_and_rows(w, ids, P, L, plan, weights, proj):
    ids_d = torch.from_numpy(ids).cuda()
    idx = plan.hash(ids_d, proj)
    e = plan.gather(idx, weights.table, weights.scales)
    xp = O.project(ids, P)
    z = O.hash_heads(xp, L.multipliers, L.primes, w.N, w.K).reshape(-1, w.R)
    assert np.array_equal(idx.cpu().numpy(), z)
    for lo in range(0, z.shape[0], CHUNK):
        hi = min(z.shape[0], lo + CHUNK)
        ref = O.gather_concat(z[lo:hi], L.tables(), w.table_dtype, L.table_scales())
        got = bf16_bits(e[lo:hi])
        assert np.array_equal(got, O.f64_to_bf16_bits(ref)), lo
    return idx, e


def sample_positions(w, n_random=64, seed=0):
    rng = np.random.default_rng(seed)
    pos = {(b, t) for b in range(w.B) for t in (0, 1, 2, 3, w.T - 1)}
    pos |= {(int(rng.integers(w.B)), int(rng.integers(w.T))) for _ in range(n_random)}
    return sorted(pos)


def check_sampled(w, ids, P, L, H_out, positions):
    ref = O.forward_at(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, positions)
    got = np.stack([act_to_f64(H_out[b, t]) for b, t in positions])
    assert_close(got, ref, w.act_dtype, w.name)


def test_tiny_f32_full():
    w = W.TINY_F32
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 0)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)
    assert np.array_equal(idx.cpu().numpy(), ref["z"].reshape(-1, w.R))
    e = plan.gather(idx, weights.table)
    assert np.array_equal(e.cpu().numpy(), ref["e"].reshape(-1, w.d_mem).astype(np.float32))
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    assert_close(act_to_f64(H), ref["H_new"], "f32", w.name)


@pytest.mark.parametrize("layer", W.PREFILL_BF16.layers)
def test_prefill_bf16_full(layer):
    w = W.PREFILL_BF16
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, layer)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    check_indices_and_rows(w, ids, P, L, plan, weights, proj)
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    assert plan.get_error() == (0, 0)
    ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)["H_new"]
    assert_close(act_to_f64(H), ref, "bf16", f"{w.name} layer {layer}")


@pytest.mark.parametrize("layer", W.DECODE_BF16.layers)
def test_decode_bf16_full(layer):
    w = W.DECODE_BF16
    T_all = w.prefix_len + 1
    ids = W.token_stream(w, T=T_all)
    P = W.projection_map(w)
    L = W.layer_inputs(w, layer, T=T_all)
    plan, weights, proj, H = make_layer(w, L, P, w.B * T_all)
    ids_d = torch.from_numpy(ids).cuda()
    st = EngramState.zeros(plan, w.B)
    pre = H[:, :w.prefix_len].contiguous()
    plan.forward(ids_d[:, :w.prefix_len].contiguous(), proj, weights, pre, st)
    step = H[:, w.prefix_len:].contiguous()
    plan.forward(ids_d[:, w.prefix_len:].contiguous(), proj, weights, step, st)
    assert plan.get_error() == (0, 0)
    ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)["H_new"]
    assert_close(act_to_f64(step), ref[:, w.prefix_len:], "bf16", "decode step")
    assert_close(act_to_f64(pre), ref[:, :w.prefix_len], "bf16", "prefix")


def test_int8_host_full():
    w = W.INT8_HOST
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, w.layers[0])
    plan, weights, proj, H = make_layer(w, L, P, ids.size)          # HBM copy of the table
    idx, e_hbm = check_indices_and_rows(w, ids, P, L, plan, weights, proj)
    table_host = to_torch(L.table, "i8", "cpu", pin=True)
    e_uva = plan.gather(idx, table_host, weights.scales)
    assert torch.equal(e_uva.view(torch.int16), e_hbm.view(torch.int16))
    H_uva = H.clone()
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    weights.table = table_host
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H_uva)
    assert plan.get_error() == (0, 0)
    assert torch.equal(H.view(torch.int16), H_uva.view(torch.int16))
    check_sampled(w, ids, P, L, H, sample_positions(w))


def test_multibranch_n4_full():
    w = W.MULTIBRANCH_N4
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, w.layers[0])
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    check_indices_and_rows(w, ids, P, L, plan, weights, proj)
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    assert plan.get_error() == (0, 0)
    check_sampled(w, ids, P, L, H, sample_positions(w, n_random=48))
