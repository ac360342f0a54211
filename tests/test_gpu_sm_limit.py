"""Stage B's persistent kernels limited to fewer SMs (engram_plan_set_sm_limit)
and a host-table gather on a chosen number of SMs (engram_plan_set_host_gather_sms)
give the same bits as the defaults; a batch in pieces -- each piece's Stage A
over host-memory tables on one stream, beside the previous piece's Stage B on
another -- equals one call, on plain streams and on the two groups of an SM
split (engram_sm_split_*)."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from hashed_gram_embedding_engram_gb300 import EngramError, SmSplit  # noqa: E402
from tests.gpu_helpers import make_layer, to_torch  # noqa: E402

BF16 = W.PREFILL_BF16.scaled(V=5000, V_proj=3850, prime_target=4001)
I8 = W.INT8_HOST.scaled(B=8, T=600, V=5000, V_proj=3850, prime_target=3001, span_copies=3)


def bits(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("B,T,limit,pairs", [(1, 4096, 114, False), (2, 1300, 37, False), (3, 500, 1, False),
                                             (1, 2600, 0, False), (2, 2048, 37, True), (1, 1024, 1, True)])
def test_sm_limit_keeps_the_bits(B, T, limit, pairs):
    w = BF16.scaled(B=B, T=T)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    ref = H0.clone()
    plan.forward(ids_d, proj, weights, ref)
    plan.set_cta_pairs(pairs)
    plan.set_sm_limit(limit)
    got = H0.clone()
    plan.forward(ids_d, proj, weights, got)
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(got), bits(ref))


def run_pieces(plan, weights, proj, ids_d, table_host, H, pieces, sa, sb, T, d_mem):
    es = [torch.empty((hi - lo) * T, d_mem, dtype=torch.bfloat16, device="cuda") for lo, hi in pieces]
    cur = torch.cuda.current_stream()
    sa.wait_stream(cur)
    sb.wait_stream(cur)
    ready = []
    with torch.cuda.stream(sa):
        for (lo, hi), ep in zip(pieces, es):
            plan.stage_a(ids_d[lo:hi], proj, table_host, weights.scales, out=ep)
            ev = torch.cuda.Event()
            ev.record(sa)
            ready.append(ev)
    with torch.cuda.stream(sb):
        for (lo, hi), ep, ev in zip(pieces, es, ready):
            sb.wait_event(ev)
            plan.stage_b(ep, weights, H[lo:hi])
    cur.wait_stream(sa)
    cur.wait_stream(sb)
    torch.cuda.synchronize()


@pytest.mark.parametrize("split", [False, True])
def test_pieces_beside_a_host_table_lookup_equal_one_call(split):
    w = I8
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size)
    table_host = to_torch(L.table, "i8", "cpu", pin=True)
    ids_d = torch.from_numpy(ids).cuda()
    ref = H0.clone()
    e = plan.stage_a(ids_d, proj, table_host, weights.scales)
    plan.stage_b(e, weights, ref)
    n_dev = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan.host_gather_sms() == n_dev // 4
    pieces = [(0, 3), (3, 5), (5, 8)]
    H = H0.clone()
    if split:
        sp = SmSplit(16)
        assert sp.sms[0] >= 16 and sp.sms[0] + sp.sms[1] <= n_dev and sp.sms[1] > 0
        plan.set_host_gather_sms(sp.sms[0])
        plan.set_sm_limit(sp.sms[1])
        assert plan.host_gather_sms() == sp.sms[0]
        run_pieces(plan, weights, proj, ids_d, table_host, H, pieces, sp.stream(0), sp.stream(1), w.T, w.d_mem)
        sp.close()
    else:
        plan.set_sm_limit(n_dev - plan.host_gather_sms())
        run_pieces(plan, weights, proj, ids_d, table_host, H, pieces, torch.cuda.Stream(),
                   torch.cuda.current_stream(), w.T, w.d_mem)
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(H), bits(ref))


@pytest.mark.parametrize("n", [1, 8, 37, 500])
def test_host_gather_sms_keeps_the_bits(n):
    w = I8
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, _ = make_layer(w, L, P, ids.size)
    table_host = to_torch(L.table, "i8", "cpu", pin=True)
    ids_d = torch.from_numpy(ids).cuda()
    ref = plan.stage_a(ids_d, proj, table_host, weights.scales)
    plan.set_host_gather_sms(n)
    n_dev = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan.host_gather_sms() == min(n, n_dev)
    got = plan.stage_a(ids_d, proj, table_host, weights.scales)
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(got), bits(ref))
    plan.set_host_gather_sms(0)
    assert plan.host_gather_sms() == n_dev // 4


def test_split_argument_errors():
    n_dev = torch.cuda.get_device_properties(0).multi_processor_count
    for n in (0, -3, n_dev, n_dev + 8):
        with pytest.raises(EngramError):
            SmSplit(n)
    w = BF16
    L = W.layer_inputs(w, 1)
    plan, *_ = make_layer(w, L, W.projection_map(w), 64)
    with pytest.raises(EngramError):
        plan.set_sm_limit(-1)
    with pytest.raises(EngramError):
        plan.set_host_gather_sms(-1)


# ---------------------------------------------------------------- engram_forward_split
def _layer(w, host):
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size, table_on_host=host)
    return plan, weights, proj, H0, torch.from_numpy(ids).cuda()


@pytest.fixture(scope="module")
def split():
    sp = SmSplit(16)
    yield sp
    sp.close()


@pytest.mark.parametrize("host,n_pieces", [(True, 1), (True, 3), (True, 8), (False, 2)])
def test_forward_split_equals_forward(split, host, n_pieces):
    w = I8 if host else BF16.scaled(B=4, T=700)
    plan, weights, proj, H0, ids_d = _layer(w, host)
    ref = H0.clone()
    plan.forward(ids_d, proj, weights, ref)
    plan.set_sm_limit(100)
    plan.set_host_gather_sms(5)
    got = H0.clone()
    plan.forward_split(split, n_pieces, ids_d, proj, weights, got)
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(got), bits(ref))
    assert plan.host_gather_sms() == 5               # the plan's own settings are back


def test_forward_split_continues_sequences_with_state(split):
    """Two chunks of every sequence: the second through the split with the state
    the first left, against two plain forwards (H and the whole state, bit for bit)."""
    w = I8.scaled(B=6, T=400)
    plan, weights, proj, H0, ids_d = _layer(w, True)
    from hashed_gram_embedding_engram_gb300 import EngramState
    st_ref, st = EngramState.zeros(plan, w.B), EngramState.zeros(plan, w.B)
    ref, got = H0.clone(), H0.clone()
    plan.forward(ids_d, proj, weights, ref, st_ref)
    plan.forward(ids_d, proj, weights, got, st)
    ids2 = torch.flip(ids_d, dims=[1]).contiguous()
    ref2, got2 = H0.clone(), H0.clone()
    plan.forward(ids2, proj, weights, ref2, st_ref)
    plan.forward_split(split, 4, ids2, proj, weights, got2, st)
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(got2), bits(ref2))
    for a, b in ((st.prev_ids, st_ref.prev_ids), (st.u_ring, st_ref.u_ring), (st.pos, st_ref.pos)):
        assert torch.equal(a, b)


def test_forward_split_in_a_cuda_graph(split):
    w = I8
    plan, weights, proj, H0, ids_d = _layer(w, True)
    ref = H0.clone()
    plan.forward(ids_d, proj, weights, ref)
    H = H0.clone()
    ws = plan.new_workspace(ids_d.numel(), "cuda")
    plan.forward_split(split, 4, ids_d, proj, weights, H, workspace=ws)     # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.forward_split(split, 4, ids_d, proj, weights, H, workspace=ws)
    for _ in range(2):
        H.copy_(H0)
        g.replay()
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(H), bits(ref))


def test_forward_split_argument_errors(split):
    w = I8.scaled(B=3, T=64)
    plan, weights, proj, H0, ids_d = _layer(w, True)
    for n in (0, 4, 65):
        with pytest.raises(EngramError):
            plan.forward_split(split, n, ids_d, proj, weights, H0.clone())
    assert plan.get_error() == (0, 0)


def test_forward_split_through_the_hot_row_cache(split):
    """Every piece's Stage A through an LFU-built HBM cache of the host table:
    the bits of the plain forward, and the cache's counters see every lookup."""
    from hashed_gram_embedding_engram_gb300 import EngramCache
    w = I8
    plan, weights, proj, H0, ids_d = _layer(w, True)
    ref = H0.clone()
    plan.forward(ids_d, proj, weights, ref)
    cache = EngramCache(plan, max(1, plan.total_rows // 20), weights.table)
    cache.observe(torch.from_numpy(W.token_stream(w, key="cache-warm")).cuda(), proj)
    assert cache.build() > 0
    cache.stats(reset=True)
    got = H0.clone()
    plan.forward_split(split, 4, ids_d, proj, weights, got, cache=cache)
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(got), bits(ref))
    looked, hits, link, _ = cache.stats()
    assert looked == ids_d.numel() * plan.R and 0 < hits < looked and link == looked - hits
    # the per-batch dedup runs its own pipeline; a cache of another plan is refused
    cache.set_dedup(ids_d.numel() * plan.R)
    with pytest.raises(EngramError):
        plan.forward_split(split, 4, ids_d, proj, weights, H0.clone(), cache=cache)
    cache.set_dedup(0)
    other, *_ = _layer(w, True)
    with pytest.raises(EngramError):
        other.forward_split(split, 4, ids_d, proj, weights, H0.clone(), cache=cache)
    cache.close()


@pytest.mark.parametrize("name", ["tiny_f32", "small_multibranch"])
def test_forward_split_other_shapes(split, name):
    """fp32 layers (SIMT projection, gate kernel) and four branches (M = 4, the
    finalize kernel): the split form equals the plain forward bit for bit."""
    w = {"tiny_f32": W.TINY_F32.scaled(B=3),
         "small_multibranch": W.MULTIBRANCH_N4.scaled(B=3, T=129, V=5000, V_proj=3850, prime_target=2003, d=256,
                                                      span_copies=3)}[name]
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, w.layers[0])
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size, table_on_host=True)
    ids_d = torch.from_numpy(ids).cuda()
    ref = H0.clone()
    plan.forward(ids_d, proj, weights, ref)
    got = H0.clone()
    plan.forward_split(split, min(2, w.B), ids_d, proj, weights, got)
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    view = (lambda t: t.contiguous().view(torch.int32)) if w.act_dtype == "f32" else bits
    assert torch.equal(view(got), view(ref))


@pytest.mark.parametrize("name", ["small_i8", "small_multibranch"])
def test_forward_split_matches_oracle(split, name):
    """engram_forward_split's H against the float64 oracle (Steps 1-8), element by
    element, within the bf16 tolerance."""
    from oracle import engram_oracle as O
    from tests.gpu_helpers import act_to_f64, assert_close
    from tests.test_gpu_parity import SMALL
    w = SMALL[name]
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, w.layers[0])
    ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, None)
    plan, weights, proj, H = make_layer(w, L, P, ids.size, table_on_host=True)
    plan.forward_split(split, w.B, torch.from_numpy(ids).cuda(), proj, weights, H)
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    assert_close(act_to_f64(H), ref["H_new"], w.act_dtype, name)


def test_forward_split_with_the_e4m3_projection(split):
    """e4m3 weights: every piece's gather writes its codes (as engram_forward's
    does); the same bits as the plain forward."""
    import dataclasses
    w = BF16.scaled(B=4, T=333)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size, table_on_host=True)
    q, sc = plan.quantize_fp8(weights.w_kv)
    w8 = dataclasses.replace(weights, w_kv=None, w_kv_fp8=q, w_kv_scale=sc)
    ids_d = torch.from_numpy(ids).cuda()
    ref = H0.clone()
    plan.forward(ids_d, proj, w8, ref)
    got = H0.clone()
    plan.forward_split(split, 3, ids_d, proj, w8, got)
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(got), bits(ref))
