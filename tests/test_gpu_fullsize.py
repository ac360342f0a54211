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
    assert_rows_equal_oracle(w, z, L, e)
    return idx, e


def oracle_rows_bits(w, z, L):
    """The oracle's gathered rows (Step 4) of indices z as bf16 bits, built in blocks."""
    out = np.empty((z.shape[0], w.d_mem), dtype=np.uint16)
    for lo in range(0, z.shape[0], CHUNK):
        hi = min(z.shape[0], lo + CHUNK)
        out[lo:hi] = O.f64_to_bf16_bits(O.gather_concat(z[lo:hi], L.tables(), w.table_dtype, L.table_scales()))
    return out


def assert_rows_equal_oracle(w, z, L, e):
    """e (the GPU's gathered rows of indices z) equals the oracle's, bit for bit, in blocks."""
    for lo in range(0, z.shape[0], CHUNK):
        hi = min(z.shape[0], lo + CHUNK)
        ref = O.gather_concat(z[lo:hi], L.tables(), w.table_dtype, L.table_scales())
        assert np.array_equal(bf16_bits(e[lo:hi]), O.f64_to_bf16_bits(ref)), lo


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


def test_prefill_graph_step_full():
    """The prefill step in the launch configuration the benchmark times: both
    layers' Stage A on a side stream, each layer's Stage B on the main stream
    once its rows are in, the whole step captured in a CUDA graph and replayed
    with H restored in between.  Every replay equals the layer-by-layer forward
    bit for bit, and the oracle at sampled positions."""
    w = W.PREFILL_BF16
    ids, P = W.token_stream(w), W.projection_map(w)
    Ls = [W.layer_inputs(w, lid) for lid in w.layers]
    built = [make_layer(w, L, P, ids.size) for L in Ls]
    ids_d = torch.from_numpy(ids).cuda()
    want = []
    for plan, weights, proj, H in built:
        Hr = H.clone()
        plan.forward(ids_d, proj, weights, Hr)
        want.append(Hr)
    H0 = [H.clone() for *_, H in built]
    es = [torch.empty(ids.size, w.d_mem, dtype=torch.bfloat16, device="cuda") for _ in built]
    wss = [plan.new_workspace(ids.size, torch.device("cuda")) for plan, *_ in built]
    side = torch.cuda.Stream()

    def step():
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        ready = []
        with torch.cuda.stream(side):
            for (plan, weights, proj, _), e in zip(built, es):
                plan.stage_a(ids_d, proj, weights.table, weights.scales, out=e)
                ev = torch.cuda.Event()
                ev.record(side)
                ready.append(ev)
        for (plan, weights, _, H), e, ev, ws in zip(built, es, ready, wss):
            main.wait_event(ev)
            plan.stage_b(e, weights, H, workspace=ws)

    def restore():
        for (*_, H), h0 in zip(built, H0):
            H.copy_(h0)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        step()
    torch.cuda.synchronize()
    for _ in range(2):
        restore()
        g.replay()
        torch.cuda.synchronize()
        for (plan, *_, H), Hr in zip(built, want):
            assert plan.get_error() == (0, 0)
            assert torch.equal(H.view(torch.int16), Hr.view(torch.int16))
    for L, (*_, H) in zip(Ls, built):
        check_sampled(w, ids, P, L, H, sample_positions(w))


@pytest.mark.parametrize("wname", ["prefill_bf16", "multibranch_n4"])
def test_fp8_projection_full(wname):
    """The e4m3 projection at full size: the weight codes and scales equal the
    oracle's byte for byte, and the layer output matches the oracle's FP8
    evaluation at sampled positions."""
    import dataclasses
    w = W.PREFILL_BF16 if wname == "prefill_bf16" else W.MULTIBRANCH_N4
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, w.layers[0])
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    q, sc = plan.quantize_fp8(weights.w_kv)
    q_ref, s_ref = O.quantize_rows_e4m3(O.widen(L.W_kv, "bf16"))
    assert np.array_equal(q.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy(), q_ref)
    assert np.array_equal(sc.cpu().numpy().astype(np.float64), s_ref)
    w8 = dataclasses.replace(weights, w_kv=None, w_kv_fp8=q, w_kv_scale=sc)
    plan.forward(torch.from_numpy(ids).cuda(), proj, w8, H)
    assert plan.get_error() == (0, 0)
    pos = sample_positions(w, n_random=48)
    ref = O.forward_at(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, pos, projection="fp8")
    got = np.stack([act_to_f64(H[b, t]) for b, t in pos])
    assert_close(got, ref, "bf16", f"{wname} fp8")


def test_int8_host_cache_and_dedup_full():
    """Stage A over the host link at full size with the HBM hot-row cache, the
    per-batch dedup and both: every output equals the oracle's gathered rows
    (Steps 1-4) bit for bit, in full; with the dedup every lookup is served from HBM and each distinct uncached
    row (the oracle's count when nothing is cached) crosses the link once."""
    from hashed_gram_embedding_engram_gb300 import EngramCache
    w = W.INT8_HOST
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, w.layers[0])
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    table_host = to_torch(L.table, "i8", "cpu", pin=True)
    ids_d = torch.from_numpy(ids).cuda()
    ref = plan.stage_a(ids_d, proj, table_host, weights.scales)
    z = O.hash_heads(O.project(ids, P), L.multipliers, L.primes, w.N, w.K).reshape(-1, w.R)
    oracle_bits = oracle_rows_bits(w, z, L)
    assert np.array_equal(bf16_bits(ref), oracle_bits)
    offsets = np.concatenate([[0], np.cumsum(np.asarray(L.primes, dtype=np.int64))[:-1]])
    uniq = len(np.unique(z.astype(np.int64) + offsets[None, :]))
    n = ids.size * w.R
    warm = torch.from_numpy(W.token_stream(w, key="cache-warm")).cuda()
    for capacity, dedup in ((0, True), (int(0.05 * plan.total_rows), False), (int(0.05 * plan.total_rows), True)):
        c = EngramCache(plan, capacity, table_host)
        if capacity:
            c.observe(warm, proj)
            assert c.build() > 0
        if dedup:
            c.set_dedup(n)
        c.stats(reset=True)
        got = c.stage_a(ids_d, proj, weights.scales)
        assert np.array_equal(bf16_bits(got), oracle_bits), (capacity, dedup)
        looked, from_hbm, link, _ = c.stats(reset=True)
        assert looked == n
        if dedup:
            assert from_hbm == n
            assert link == uniq if capacity == 0 else 0 < link < uniq
        else:
            assert 0 < from_hbm < n and link == n - from_hbm
        c.close()
    assert plan.get_error() == (0, 0)
