"""FP8 (e4m3) K/V projection through the C ABI against the oracle's FP8 path.

The codes and scales of the per-row quantisation are compared bit for bit
(byte work); layer outputs against the oracle's float64 evaluation of the same
quantised operands, with the bf16 tolerance of the other parity tests."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import engram_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from tests.gpu_helpers import act_to_f64, assert_close, make_layer  # noqa: E402

SMALL_BF16 = W.PREFILL_BF16.scaled(B=3, T=333, V=5000, V_proj=3850, prime_target=4001, d=256)
SMALL_MB = W.MULTIBRANCH_N4.scaled(B=2, T=257, V=5000, V_proj=3850, prime_target=2003, d=256, span_copies=3)


def fp8_layer(w, L, P, max_tokens):
    plan, weights, proj, H = make_layer(w, L, P, max_tokens)
    q, sc = plan.quantize_fp8(weights.w_kv)
    w8 = dataclasses.replace(weights, w_kv=None, w_kv_fp8=q, w_kv_scale=sc)
    return plan, w8, weights, proj, H


def test_quantize_codes_and_scales_are_the_oracles():
    from hashed_gram_embedding_engram_gb300 import EngramPlan  # noqa: F401
    w = SMALL_BF16
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, W.projection_map(w), 16)
    rng = np.random.default_rng(17)
    x = rng.standard_normal((37, 1024)) * rng.choice([1e-4, 1e-2, 1, 30, 400], (37, 1))
    x[3] = 0.0                                   # all-zero row
    x[4, :] = 1e-30                              # amax far below the e4m3 range
    x[5, 7] = 448.0 * 8                          # one dominant value
    bits = W.gen.f32_to_bf16_bits(x.astype(np.float32))
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    q, sc = plan.quantize_fp8(xb)
    xr = O.bf16_to_f64(bits)
    q_ref, s_ref = O.quantize_rows_e4m3(xr)
    got = q.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()
    assert np.array_equal(got, q_ref)
    assert np.array_equal(sc.cpu().numpy().astype(np.float64), s_ref)
    # the weights of a layer, as the forward uses them
    qw, sw = plan.quantize_fp8(weights.w_kv)
    qw_ref, sw_ref = O.quantize_rows_e4m3(O.widen(L.W_kv, "bf16"))
    assert np.array_equal(qw.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy(), qw_ref)
    assert np.array_equal(sw.cpu().numpy().astype(np.float64), sw_ref)


@pytest.mark.parametrize("w", [SMALL_BF16, SMALL_MB], ids=["small_bf16", "small_multibranch"])
def test_fp8_forward_matches_the_fp8_oracle(w):
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, projection="fp8")
    exact = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)
    plan, w8, wbf, proj, H = fp8_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    H8 = H.clone()
    plan.forward(ids_d, proj, w8, H8)
    assert plan.get_error() == (0, 0)
    assert_close(act_to_f64(H8), ref["H_new"], "bf16", "fp8")
    # it is the FP8 path that ran: closer to the FP8 oracle than to the exact one
    e8 = np.abs(act_to_f64(H8) - ref["H_new"]).mean()
    ex = np.abs(act_to_f64(H8) - exact["H_new"]).mean()
    assert e8 < ex
    # Stage A then Stage B with the same weights gives the same bits
    e = plan.stage_a(ids_d, proj, wbf.table, wbf.scales)
    H2 = H.clone()
    plan.stage_b(e, w8, H2)
    assert torch.equal(H2.view(torch.int16), H8.view(torch.int16))


def test_fp8_streaming_and_decode_are_bit_identical_to_prefill():
    """2560 tokens at d = 1024 (256-column projection tiles) against chunks of
    100 (64-column tiles) and single-token decode steps: per-token and per-row
    scales do not depend on the chunking, and the gate's sums have the same
    bits for every tile width."""
    from hashed_gram_embedding_engram_gb300 import EngramState
    w = W.PREFILL_BF16.scaled(B=1, T=2560, V=5000, V_proj=3850, prime_target=4001)
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, w8, _, proj, H = fp8_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    full = H.clone()
    plan.forward(ids_d, proj, w8, full)
    st = EngramState.zeros(plan, w.B)
    out = H.clone()
    t0 = 0
    for n in [100] * 25 + [1] * 20 + [40]:
        seg = out[:, t0:t0 + n].contiguous()
        plan.forward(ids_d[:, t0:t0 + n].contiguous(), proj, w8, seg, st)
        out[:, t0:t0 + n] = seg
        t0 += n
    assert t0 == w.T
    assert plan.get_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))
    pos = [(0, t) for t in (0, 1, 2, 9, 127, 128, 1000, 2047, 2048, 2540, 2559)]
    ref = O.forward_at(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, pos, projection="fp8")
    got = np.stack([act_to_f64(full[b, t]) for b, t in pos])
    assert_close(got, ref, "bf16", "fp8 sampled")


# ---------------------------------------------------------------- codes written by the gather
def _codes_ref(w, ids, P, L, prev=None):
    """The oracle's e4m3 codes and scales of the oracle's gathered rows."""
    from tests.test_gpu_parity import expected_e_bits
    z = O.hash_heads(O.project(ids, P), L.multipliers, L.primes, w.N, w.K, prev)
    e_bits = expected_e_bits(w, z.reshape(-1, w.R), L)
    return O.quantize_rows_e4m3(O.bf16_to_f64(e_bits.reshape(-1, w.d_mem)))


@pytest.mark.parametrize("host", [False, True])
def test_stage_a_e4m3_is_the_quantised_stage_a(host):
    """engram_stage_a_e4m3's codes and scales: byte for byte what quantize_fp8
    makes of stage_a's rows, and the oracle's quantisation of its rows; two
    layers in one launch, with state ids, give each layer's."""
    from hashed_gram_embedding_engram_gb300 import stage_a_layers_e4m3
    from tests.gpu_helpers import to_torch
    w = SMALL_BF16.scaled(B=5, T=91)
    ids, P = W.token_stream(w), W.projection_map(w)
    Ls = [W.layer_inputs(w, lid) for lid in (1, 15)]
    built = [make_layer(w, L, P, ids.size) for L in Ls]
    ids_d = torch.from_numpy(ids).cuda()
    rng = np.random.default_rng(3)
    prev = [rng.integers(0, w.V_proj, size=(w.B, w.N - 1)).astype(np.int32) for _ in Ls]
    prev_d = [torch.from_numpy(p).cuda() for p in prev]
    tables = [to_torch(L.table, "bf16", "cpu", pin=True) if host else b[1].table for L, b in zip(Ls, built)]
    outs = stage_a_layers_e4m3([b[0] for b in built], ids_d, built[0][2], tables, prev_ids=prev_d)
    for (plan, weights, proj, _), L, (q, sc), tab, pv, pvd in zip(built, Ls, outs, tables, prev, prev_d):
        e = plan.stage_a(ids_d, proj, tab, prev_ids=pvd)
        q_ref, sc_ref = plan.quantize_fp8(e)
        assert torch.equal(q, q_ref) and torch.equal(sc, sc_ref)
        q_o, s_o = _codes_ref(w, ids, P, L, pv)
        assert np.array_equal(q.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy(), q_o)
        assert np.array_equal(sc.cpu().numpy().astype(np.float64), s_o)
        assert plan.get_error() == (0, 0)


def test_stage_b_e4m3_and_forward_equal_the_quantising_stage_b():
    """Stage B from the gather's codes, and engram_forward (whose gather now
    writes the codes), give the bits of stage_a + stage_b with the separate
    quantisation launch."""
    w = SMALL_BF16
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, w8, _, proj, H0 = fp8_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    ref = H0.clone()
    plan.stage_b(plan.stage_a(ids_d, proj, w8.table), w8, ref)
    got_b = H0.clone()
    q, sc = plan.stage_a_e4m3(ids_d, proj, w8.table)
    plan.stage_b_e4m3(q, sc, w8, got_b)
    got_f = H0.clone()
    plan.forward(ids_d, proj, w8, got_f)
    assert plan.get_error() == (0, 0)
    for got in (got_b, got_f):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_e4m3_gather_refuses_what_it_does_not_cover():
    from hashed_gram_embedding_engram_gb300 import EngramError
    # 24 rows of 128 bytes: 192 chunks per token, more than one round of loads
    w = SMALL_MB
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, w8, _, proj, H0 = fp8_layer(w, L, P, ids.size)
    with pytest.raises(EngramError):
        plan.stage_a_e4m3(torch.from_numpy(ids).cuda(), proj, w8.table)
    # int8 tables
    wi = W.INT8_HOST.scaled(B=2, T=50, V=5000, V_proj=3850, prime_target=3001, d=256, span_copies=2)
    idi, Pi, Li = W.token_stream(wi), W.projection_map(wi), W.layer_inputs(wi, 1)
    pi, wti, proji, _ = make_layer(wi, Li, Pi, idi.size)
    with pytest.raises(EngramError):
        pi.stage_a_e4m3(torch.from_numpy(idi).cuda(), proji, wti.table)
    # Stage B from codes needs the FP8 weights
    w = SMALL_BF16
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size)
    q, sc = plan.stage_a_e4m3(torch.from_numpy(ids).cuda(), proj, weights.table)
    with pytest.raises(EngramError):
        plan.stage_b_e4m3(q, sc, weights, H0.clone())
    assert plan.get_error() == (0, 0)
