"""GPU path (through the C ABI) against the CPU oracle on the same seeded inputs.

Indices and gathered rows: bit-exact.  Layer outputs: max-abs 2e-2 and
relative L2 5e-3 for bf16 (fp32 accumulation), tighter for the fp32 workload.
Small cases span several 128-row GEMM tiles with ragged tails and run the
oracle in full; the full-size workloads are checked in full for the integer
work and on sampled positions (every sequence start included) for the layer
output, via the oracle's windowed evaluator.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import engram_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from tests.gpu_helpers import act_to_f64, assert_close, bf16_bits, make_layer, to_torch  # noqa: E402


SMALL = {
    "tiny_f32": W.TINY_F32,
    "small_bf16": W.PREFILL_BF16.scaled(B=3, T=333, V=5000, V_proj=3850, prime_target=4001, d=256),
    "small_i8": W.INT8_HOST.scaled(B=2, T=300, V=5000, V_proj=3850, prime_target=3001, d=256, span_copies=3),
    "small_multibranch": W.MULTIBRANCH_N4.scaled(B=2, T=257, V=5000, V_proj=3850, prime_target=2003, d=256,
                                                 span_copies=3),
}


def oracle_forward(w, ids, P, L, state=None):
    return O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, state)


def expected_e_bits(w, z, L):
    """What the gather must write, exactly: the stored rows (copy) or bf16(q*s)."""
    e = O.gather_concat(z, L.tables(), w.table_dtype, L.table_scales())
    if w.table_dtype == "f32":
        return e.astype(np.float32)
    if w.table_dtype == "bf16":
        return O.f64_to_bf16_bits(e)
    return O.f64_to_bf16_bits(e)


def gpu_e_bits(w, e):
    return e.cpu().numpy() if w.table_dtype == "f32" else bf16_bits(e)


@pytest.fixture(scope="module", params=list(SMALL))
def small(request):
    w = SMALL[request.param]
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, w.layers[0])
    ref = oracle_forward(w, ids, P, L)
    return request.param, w, ids, P, L, ref


def test_small_hash_bitexact(small):
    name, w, ids, P, L, ref = small
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    assert np.array_equal(idx.cpu().numpy(), ref["z"].reshape(-1, w.R))


def test_small_gather_bitexact(small):
    name, w, ids, P, L, ref = small
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    z = torch.from_numpy(ref["z"].reshape(-1, w.R).astype(np.int32)).cuda()
    e = plan.gather(z, weights.table, weights.scales)
    assert np.array_equal(gpu_e_bits(w, e), expected_e_bits(w, ref["z"].reshape(-1, w.R), L).reshape(e.shape))


def test_small_kv_projection(small):
    name, w, ids, P, L, ref = small
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    # exact e as the GPU stores it, then the GEMM alone
    e_bits = expected_e_bits(w, ref["z"].reshape(-1, w.R), L)
    e = to_torch(e_bits, "f32" if w.table_dtype == "f32" else "bf16")
    kv = plan.kv_projection(e, weights.w_kv)
    e64 = O.widen(e_bits, w.act_dtype)
    Wm = O.widen(L.W_kv, w.act_dtype)
    exp = e64 @ Wm.T
    got = act_to_f64(kv)
    rms = np.sqrt(np.mean(exp ** 2))
    if w.act_dtype == "bf16":
        # one bf16 rounding of an fp32 accumulation: |err| <= 2^-8 |x| plus accumulation noise
        assert np.all(np.abs(got - exp) <= 2.0 ** -8 * np.abs(exp) + 1e-3 * rms)
    else:
        assert np.all(np.abs(got - exp) <= 1e-5 * rms + 1e-6 * np.abs(exp))


def test_small_forward_matches_oracle(small):
    name, w, ids, P, L, ref = small
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    st, flags = plan.get_error()
    assert st == 0 and flags == 0
    assert_close(act_to_f64(H), ref["H_new"], w.act_dtype, name)


def test_small_stage_a_then_stage_b_matches_forward(small):
    name, w, ids, P, L, ref = small
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    idx = plan.hash(ids_d, proj)
    e = plan.gather(idx, weights.table, weights.scales)
    H2 = H.clone()
    plan.stage_b(e, weights, H2)
    plan.forward(ids_d, proj, weights, H)
    assert torch.equal(H, H2)


def test_small_stage_a_equals_hash_then_gather(small):
    name, w, ids, P, L, ref = small
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    e_fused = plan.stage_a(ids_d, proj, weights.table, weights.scales)
    e_split = plan.gather(plan.hash(ids_d, proj), weights.table, weights.scales)
    assert torch.equal(e_fused.view(torch.int8), e_split.view(torch.int8))
    H2 = H.clone()
    plan.stage_b(e_fused, weights, H2)
    plan.forward(ids_d, proj, weights, H)
    assert torch.equal(H, H2)


def test_prefetched_stage_a_on_a_side_stream_matches_forward():
    """Stage A of the second layer runs on another stream while the first layer's
    Stage B runs; the results equal two sequential forwards bit for bit."""
    w = SMALL["small_bf16"]
    ids = W.token_stream(w)
    P = W.projection_map(w)
    layers = [W.layer_inputs(w, lid) for lid in (1, 15)]
    built = [make_layer(w, L, P, ids.size) for L in layers]
    ids_d = torch.from_numpy(ids).cuda()
    ref = []
    for plan, weights, proj, H in built:
        Hr = H.clone()
        plan.forward(ids_d, proj, weights, Hr)
        ref.append(Hr)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    outs = [H.clone() for _, _, _, H in built]
    es = [torch.empty(ids.size, w.d_mem, dtype=torch.bfloat16, device="cuda") for _ in built]
    side.wait_stream(main)
    done = []
    with torch.cuda.stream(side):
        for (plan, weights, proj, _), e in zip(built, es):
            plan.stage_a(ids_d, proj, weights.table, weights.scales, out=e)
            ev = torch.cuda.Event()
            ev.record(side)
            done.append(ev)
    for (plan, weights, proj, _), e, ev, Ho in zip(built, es, done, outs):
        main.wait_event(ev)
        plan.stage_b(e, weights, Ho)
    torch.cuda.synchronize()
    for Ho, Hr in zip(outs, ref):
        assert torch.equal(Ho.view(torch.int16), Hr.view(torch.int16))


def test_zero_table_leaves_H_bit_unchanged():
    w = SMALL["small_bf16"]
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    L.table[:] = 0
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    H0 = H.clone()
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    assert torch.equal(H.view(torch.int16), H0.view(torch.int16))


@pytest.mark.parametrize("T", [1, 2, 5, 129])
def test_short_and_ragged_sequences(T):
    w = SMALL["small_bf16"].scaled(B=5, T=T)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    ref = oracle_forward(w, ids, P, L)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    assert np.array_equal(idx.cpu().numpy(), ref["z"].reshape(-1, w.R))
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    assert_close(act_to_f64(H), ref["H_new"], "bf16", f"T={T}")


def test_empty_input_is_a_no_op():
    w = SMALL["small_bf16"]
    L = W.layer_inputs(w, 1)
    P = W.projection_map(w)
    plan, weights, proj, H = make_layer(w, L, P, 16)
    ids = torch.zeros(0, 7, dtype=torch.int32, device="cuda")
    Hz = torch.zeros(0, 7, 1, w.d, dtype=torch.bfloat16, device="cuda")
    plan.forward(ids, proj, weights, Hz)
    assert plan.get_error() == (0, 0)


def test_causality_on_gpu():
    w = SMALL["small_bf16"].scaled(B=1, T=200)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    H1 = H.clone()
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H1)
    ids2 = ids.copy()
    ids2[0, 120:] = (ids2[0, 120:] + 7) % w.V
    H2 = H.clone()
    H2[0, 150:] += 1.0
    plan.forward(torch.from_numpy(ids2).cuda(), proj, weights, H2)
    assert torch.equal(H1[0, :120], H2[0, :120])
    assert not torch.equal(H1[0, 120:132], H2[0, 120:132])


# --------------------------------------------------------------------------- #
# streaming: chunked prefill and decode
# --------------------------------------------------------------------------- #
def test_decode_steps_match_prefill_and_oracle():
    from hashed_gram_embedding_engram_gb300 import EngramState
    w = SMALL["small_bf16"].scaled(B=6, T=40)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    ref = oracle_forward(w, ids, P, L)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    full = H.clone()
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, full)
    st = EngramState.zeros(plan, w.B)
    ids_d = torch.from_numpy(ids).cuda()
    out = H.clone()
    prefix = 17
    chunk = out[:, :prefix].contiguous()
    plan.forward(ids_d[:, :prefix].contiguous(), proj, weights, chunk, st)
    out[:, :prefix] = chunk
    for t in range(prefix, w.T):
        step = out[:, t:t + 1].contiguous()
        plan.forward(ids_d[:, t:t + 1].contiguous(), proj, weights, step, st)
        out[:, t:t + 1] = step
    assert plan.get_error() == (0, 0)
    assert torch.equal(st.pos.cpu(), torch.full((w.B,), w.T, dtype=torch.int32))
    # the streamed result equals one-shot prefill bit for bit, and the oracle within tolerance
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))
    assert_close(act_to_f64(out), ref["H_new"], "bf16", "streamed")
    # prev ids hold the last N-1 projected ids
    assert np.array_equal(st.prev_ids.cpu().numpy(), ref["state"]["prev"])


def test_chunked_prefill_with_ragged_chunks():
    from hashed_gram_embedding_engram_gb300 import EngramState
    w = SMALL["small_multibranch"].scaled(B=2, T=61)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    full = H.clone()
    ids_d = torch.from_numpy(ids).cuda()
    plan.forward(ids_d, proj, weights, full)
    st = EngramState.zeros(plan, w.B)
    out = H.clone()
    t0 = 0
    for n in (1, 2, 3, 13, 5, 37):
        seg = out[:, t0:t0 + n].contiguous()
        plan.forward(ids_d[:, t0:t0 + n].contiguous(), proj, weights, seg, st)
        out[:, t0:t0 + n] = seg
        t0 += n
    assert t0 == w.T
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))


def test_streaming_bit_identical_across_gemm_tile_widths():
    """2560 tokens at d = 1024 give the K/V projection 20 x 8 tiles of 128 x 256
    (inside the one-launch Stage B); chunks of 100 tokens through the two-launch
    form run it with 128 x 64 tiles.  The gate's partial sums are
    combined as one pairwise tree over 32-column chunks either way, so the
    outputs agree bit for bit; the oracle checks a sample of positions."""
    from hashed_gram_embedding_engram_gb300 import EngramState
    w = W.PREFILL_BF16.scaled(B=1, T=2560, V=5000, V_proj=3850, prime_target=4001)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    full = H.clone()
    plan.set_fused_stage_b(True)
    plan.forward(ids_d, proj, weights, full)
    plan.set_fused_stage_b(False)
    st = EngramState.zeros(plan, w.B)
    out = H.clone()
    for t0 in range(0, w.T, 100):
        t1 = min(t0 + 100, w.T)
        seg = out[:, t0:t1].contiguous()
        plan.forward(ids_d[:, t0:t1].contiguous(), proj, weights, seg, st)
        out[:, t0:t1] = seg
    assert plan.get_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))
    pos = [(0, t) for t in (0, 1, 2, 9, 10, 11, 127, 128, 1000, 2047, 2048, 2559)]
    ref = O.forward_at(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, pos)
    got = np.stack([act_to_f64(full[b, t]) for b, t in pos])
    assert_close(got, ref, "bf16", "sampled")


@pytest.mark.parametrize("B,T,chunks", [(1, 333, 4), (6, 40, 4), (3, 50, 1)])
def test_layer_pipelines_host_inputs_bit_exactly(B, T, chunks):
    """EngramLayer with H in pinned host memory (pieces of the batch or of the one
    sequence copied in, computed and copied back on three streams) equals one
    device-resident forward bit for bit."""
    from hashed_gram_embedding_engram_gb300 import EngramLayer
    w = SMALL["small_bf16"].scaled(B=B, T=T)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    ref = H.clone()
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, ref)
    layer = EngramLayer(plan, weights, proj, chunks=chunks)
    ids_h = torch.from_numpy(ids).pin_memory()
    H_h = H.cpu().pin_memory()
    for _ in range(2):                        # twice: buffers and streams are reused
        out = H.cpu().pin_memory()
        layer(ids_h, out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(H_h.view(torch.int16), H.cpu().view(torch.int16))   # the caller's input untouched


def test_layer_with_state_split_along_the_batch():
    """A host-resident decode-style call split along the batch with a streaming
    state: each piece continues its own sequences' state; the result and the
    state equal one device-resident call's, bit for bit."""
    from hashed_gram_embedding_engram_gb300 import EngramLayer, EngramState
    w = SMALL["small_bf16"].scaled(B=6, T=40)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    st_ref, st = EngramState.zeros(plan, w.B), EngramState.zeros(plan, w.B)
    pre = H[:, :30].contiguous()
    plan.forward(ids_d[:, :30].contiguous(), proj, weights, pre.clone(), st_ref)
    plan.forward(ids_d[:, :30].contiguous(), proj, weights, pre.clone(), st)
    ref = H[:, 30:].contiguous()
    plan.forward(ids_d[:, 30:].contiguous(), proj, weights, ref, st_ref)
    layer = EngramLayer(plan, weights, proj, chunks=3)
    out = H[:, 30:].contiguous().cpu().pin_memory()
    layer(torch.from_numpy(ids[:, 30:].copy()).pin_memory(), out, st)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))
    for a, b in ((st.prev_ids, st_ref.prev_ids), (st.u_ring, st_ref.u_ring), (st.pos, st_ref.pos)):
        assert torch.equal(a, b)


def test_independent_layers_overlap_and_stay_bit_exact():
    """Two independent layers with host-resident H, called with one fork event
    and joined afterwards (so each one's copies overlap the other's compute),
    eagerly and replayed from a CUDA graph, three times on the same buffers:
    each equals its own device-resident forward bit for bit."""
    from hashed_gram_embedding_engram_gb300 import EngramLayer
    w = SMALL["small_bf16"].scaled(B=1, T=300)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    ids_h = torch.from_numpy(ids).pin_memory()
    lays, refs, outs, inputs = [], [], [], []
    for lid in (1, 15):
        L = W.layer_inputs(w, lid)
        plan, weights, proj, H = make_layer(w, L, P, ids.size)
        ref = H.clone()
        plan.forward(torch.from_numpy(ids).cuda(), proj, weights, ref)
        lays.append(EngramLayer(plan, weights, proj, chunks=2))
        refs.append(ref.cpu())
        inputs.append(H.cpu().pin_memory())
        outs.append(H.cpu().pin_memory())

    def step():
        fork = torch.cuda.Event()
        fork.record(torch.cuda.current_stream())
        for lay, out in zip(lays, outs):
            lay(ids_h, out, join=False, after=fork)
        for lay in lays:
            lay.join()

    def check():
        torch.cuda.synchronize()
        for out, ref in zip(outs, refs):
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16))

    for _ in range(3):
        for out, inp in zip(outs, inputs):
            out.copy_(inp)
        step()
        check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        step()
    for _ in range(3):
        for out, inp in zip(outs, inputs):
            out.copy_(inp)
        g.replay()
        check()


# --------------------------------------------------------------------------- #
# UVA: host-resident tables
# --------------------------------------------------------------------------- #
def test_uva_gather_equals_hbm_gather():
    w = SMALL["small_i8"]
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, wd, proj, H = make_layer(w, L, P, ids.size)
    table_host = to_torch(L.table, "i8", "cpu", pin=True)
    scales_host = to_torch(L.scales, "f16", "cpu", pin=True)
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    e_dev = plan.gather(idx, wd.table, wd.scales)
    e_host = plan.gather(idx, table_host, scales_host)
    e_mix = plan.gather(idx, table_host, wd.scales)
    assert torch.equal(e_dev.view(torch.int16), e_host.view(torch.int16))
    assert torch.equal(e_dev.view(torch.int16), e_mix.view(torch.int16))


# --------------------------------------------------------------------------- #
# HBM hot-row cache in front of host tables
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("kind", ["small_i8", "small_bf16"])
def test_cached_stage_a_equals_uva_and_hbm_gathers(kind):
    """Rows read through the cache are the rows of the table: the cached Stage A
    equals the oracle's gathered rows (Steps 1-4) bit for bit, before any build
    (nothing cached), after an LFU build, and with every row cached, as do the
    plain Stage A over the HBM table and over UVA; the counters see every row
    and the hits the build promised."""
    from hashed_gram_embedding_engram_gb300 import EngramCache
    w = SMALL[kind]
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, wd, proj, H = make_layer(w, L, P, ids.size)
    table_host = to_torch(L.table, w.table_dtype, "cpu", pin=True)
    ids_d = torch.from_numpy(ids).cuda()
    oracle_bits = oracle_rows_bits(w, ids, P, L)
    ref = plan.stage_a(ids_d, proj, wd.table, wd.scales)
    assert np.array_equal(bf16_bits(ref), oracle_bits.reshape(ref.shape))
    uva = plan.stage_a(ids_d, proj, table_host, wd.scales)
    assert torch.equal(ref.view(torch.int16), uva.view(torch.int16))
    n_rows = int(np.sum(L.primes))
    cache = EngramCache(plan, max(1, n_rows // 50), table_host)
    got = cache.stage_a(ids_d, proj, wd.scales)
    assert np.array_equal(bf16_bits(got), oracle_bits.reshape(got.shape))
    looked, hits, link, cached = cache.stats(reset=True)
    assert looked == ids.size * w.R and hits == 0 and cached == 0 and link == looked
    # LFU: observe a different sample of the same distribution, then serve this batch
    warm = torch.from_numpy(W.token_stream(w, key="cache-warm")).cuda()
    cache.observe(warm, proj)
    cached = cache.build()
    assert 0 < cached <= n_rows // 50
    got = cache.stage_a(ids_d, proj, wd.scales)
    assert np.array_equal(bf16_bits(got), oracle_bits.reshape(got.shape))
    looked, hits, link, _ = cache.stats(reset=True)
    assert looked == ids.size * w.R and 0 < hits < looked and link == looked - hits
    # the most-counted rows of the warm sample are cached: their accesses in it are all hits
    cache.stage_a(warm, proj, wd.scales)
    looked_w, hits_w, _, _ = cache.stats(reset=True)
    assert hits_w / looked_w >= hits / looked
    full = EngramCache(plan, n_rows, table_host)
    full.observe(ids_d, proj)
    assert full.build() == len(np.unique(ref_rows(w, ids, P, L)))
    got = full.stage_a(ids_d, proj, wd.scales)
    assert np.array_equal(bf16_bits(got), oracle_bits.reshape(got.shape))
    looked, hits, link, _ = full.stats()
    assert hits == looked and link == 0


@pytest.mark.parametrize("kind", ["small_i8", "small_bf16"])
def test_dedup_stage_a_fetches_each_row_once(kind):
    """Per-batch dedup: every distinct row of the batch crosses the host link
    once (the oracle's count of distinct rows), every lookup is served from HBM,
    and the output equals the oracle's gathered rows bit for bit -- on two batches in a
    row (the slots are released), with a batch region too small for the batch
    (no dedup then), combined with an LFU cache, and replayed from a CUDA
    graph."""
    from hashed_gram_embedding_engram_gb300 import EngramCache
    w = SMALL[kind]
    ids = W.token_stream(w)
    ids2 = W.token_stream(w, key="dedup-second")
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, wd, proj, H = make_layer(w, L, P, ids.size)
    table_host = to_torch(L.table, w.table_dtype, "cpu", pin=True)
    n = ids.size * w.R
    for batch in (ids, ids2):
        ids_d = torch.from_numpy(batch).cuda()
        oracle_bits = oracle_rows_bits(w, batch, P, L)
        ref = plan.stage_a(ids_d, proj, wd.table, wd.scales)
        assert np.array_equal(bf16_bits(ref), oracle_bits.reshape(ref.shape))
        uniq = len(np.unique(ref_rows(w, batch, P, L)))
        assert uniq < n                                        # Zipf: some rows repeat
        dd = EngramCache(plan, 0, table_host)
        dd.set_dedup(n)
        for _ in range(2):
            got = dd.stage_a(ids_d, proj, wd.scales)
            assert np.array_equal(bf16_bits(got), oracle_bits.reshape(got.shape))
            looked, from_hbm, link, cached = dd.stats(reset=True)
            assert (looked, from_hbm, link, cached) == (n, n, uniq, 0)
        # a region too small for the batch: no dedup, every lookup over the link
        dd.set_dedup(n - 1)
        got = dd.stage_a(ids_d, proj, wd.scales)
        assert np.array_equal(bf16_bits(got), oracle_bits.reshape(got.shape))
        assert dd.stats(reset=True) == (n, 0, n, 0)
        dd.close()
    # with the LFU cache: cached rows never cross the link, the others once each
    ids_d = torch.from_numpy(ids).cuda()
    oracle_bits = oracle_rows_bits(w, ids, P, L)
    ref = plan.stage_a(ids_d, proj, wd.table, wd.scales)
    n_rows = int(np.sum(L.primes))
    both = EngramCache(plan, max(1, n_rows // 50), table_host)
    both.observe(torch.from_numpy(W.token_stream(w, key="cache-warm")).cuda(), proj)
    assert both.build() > 0
    both.set_dedup(n)
    got = both.stage_a(ids_d, proj, wd.scales)
    assert np.array_equal(bf16_bits(got), oracle_bits.reshape(got.shape))
    looked, from_hbm, link, _ = both.stats(reset=True)
    uniq = len(np.unique(ref_rows(w, ids, P, L)))
    assert looked == n and from_hbm == n and 0 < link < uniq
    # captured once, replayed twice: the claim, fetch, gather and release all replay
    out = torch.empty_like(ref)
    dd = EngramCache(plan, 0, table_host)
    dd.set_dedup(n)
    dd.stage_a(ids_d, proj, wd.scales, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            dd.stage_a(ids_d, proj, wd.scales, out=out)
    torch.cuda.current_stream().wait_stream(s)
    dd.stats(reset=True)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_bits(out), oracle_bits.reshape(out.shape))
    assert dd.stats(reset=True)[2] == 2 * uniq
    assert plan.get_error() == (0, 0)


def oracle_rows_bits(w, ids, P, L):
    """The batch's gathered rows as the oracle defines them (Steps 1-4), as bf16 bits."""
    z = O.hash_heads(O.project(ids, P), L.multipliers, L.primes, w.N, w.K).reshape(-1, w.R)
    return expected_e_bits(w, z, L)


def ref_rows(w, ids, P, L):
    """Global table rows a batch reads, from the oracle's indices."""
    z = O.hash_heads(O.project(ids, P), L.multipliers, L.primes, w.N, w.K).reshape(-1, w.R)
    offsets = np.concatenate([[0], np.cumsum(L.primes)[:-1]]).astype(np.int64)
    return (z.astype(np.int64) + offsets[None, :]).ravel()
