"""Stage A of several layers in one launch (engram_stage_a_layers) against
per-layer engram_stage_a calls (bit for bit: the same kernel body per layer)
and against the oracle's gathered rows (Steps 1-4 of "DeepSeek Engram 系列导读",
section "Engram 工作原理").

Cases: the two prefill layers at a reduced size; three layers of a ragged
batch continuing sequences (per-layer state ids); int8 tables in HBM and in
pinned host memory; the timed step's form (one launch on a side stream, each
Stage B after it); argument errors.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import engram_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from hashed_gram_embedding_engram_gb300 import EngramError, stage_a_layers  # noqa: E402
from tests.gpu_helpers import bf16_bits, make_layer, to_torch  # noqa: E402
from tests.test_gpu_parity import expected_e_bits  # noqa: E402

BF16 = W.PREFILL_BF16.scaled(B=3, T=333, V=5000, V_proj=3850, prime_target=4001, d=256)
I8 = W.INT8_HOST.scaled(B=2, T=300, V=5000, V_proj=3850, prime_target=3001, d=256, span_copies=3)


def build(w, lids, ntok):
    P = W.projection_map(w)
    Ls = [W.layer_inputs(w, lid) for lid in lids]
    return P, Ls, [make_layer(w, L, P, ntok) for L in Ls]


def oracle_bits(w, ids, P, L, prev=None):
    z = O.hash_heads(O.project(ids, P), L.multipliers, L.primes, w.N, w.K, prev)
    return expected_e_bits(w, z.reshape(-1, w.R), L)


@pytest.mark.parametrize("lids", [(1, 15), (1,)])
def test_layers_equal_per_layer_stage_a_and_oracle(lids):
    w = BF16
    ids = W.token_stream(w)
    P, Ls, built = build(w, lids, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    plans = [b[0] for b in built]
    proj = built[0][2]
    outs = stage_a_layers(plans, ids_d, proj, [b[1].table for b in built])
    for (plan, weights, pr, _), L, e in zip(built, Ls, outs):
        ref = plan.stage_a(ids_d, pr, weights.table, weights.scales)
        assert np.array_equal(bf16_bits(e), bf16_bits(ref))
        assert np.array_equal(bf16_bits(e), oracle_bits(w, ids, P, L))
        assert plan.get_error() == (0, 0)


def test_three_layers_ragged_with_state_ids():
    w = BF16.scaled(B=5, T=37)
    lids = (1, 7, 15)
    ids = W.token_stream(w)
    P, Ls, built = build(w, lids, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    rng = np.random.default_rng(5)
    prev = [rng.integers(0, w.V_proj, size=(w.B, w.N - 1)).astype(np.int32) for _ in lids]
    prev_d = [torch.from_numpy(p).cuda() for p in prev]
    plans = [b[0] for b in built]
    outs = stage_a_layers(plans, ids_d, built[0][2], [b[1].table for b in built], prev_ids=prev_d)
    for (plan, weights, pr, _), L, e, pv, pvd in zip(built, Ls, outs, prev, prev_d):
        ref = plan.stage_a(ids_d, pr, weights.table, weights.scales, prev_ids=pvd)
        assert np.array_equal(bf16_bits(e), bf16_bits(ref))
        assert np.array_equal(bf16_bits(e), oracle_bits(w, ids, P, L, pv))


@pytest.mark.parametrize("host", [False, True])
def test_int8_layers(host):
    w = I8
    ids = W.token_stream(w)
    P, Ls, built = build(w, (1, 15), ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    tables = [to_torch(L.table, "i8", "cpu", pin=True) if host else b[1].table for L, b in zip(Ls, built)]
    plans = [b[0] for b in built]
    outs = stage_a_layers(plans, ids_d, built[0][2], tables, scales=[b[1].scales for b in built])
    for (plan, weights, pr, _), L, e, tab in zip(built, Ls, outs, tables):
        ref = plan.stage_a(ids_d, pr, tab, weights.scales)
        assert np.array_equal(bf16_bits(e), bf16_bits(ref))
        assert np.array_equal(bf16_bits(e), oracle_bits(w, ids, P, L))


def test_one_launch_ahead_of_every_stage_b_matches_forward():
    """The benchmark's form: every layer's rows from one launch on a side stream,
    then each layer's Stage B on the main stream -- the bits of per-layer forwards."""
    w = BF16
    ids = W.token_stream(w)
    P, Ls, built = build(w, (1, 15), ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    ref = []
    for plan, weights, proj, H in built:
        Hr = H.clone()
        plan.forward(ids_d, proj, weights, Hr)
        ref.append(Hr)
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    es = [torch.empty(ids.size, w.d_mem, dtype=torch.bfloat16, device="cuda") for _ in built]
    outs = [H.clone() for *_, H in built]
    side.wait_stream(main)
    with torch.cuda.stream(side):
        stage_a_layers([b[0] for b in built], ids_d, built[0][2], [b[1].table for b in built], outs=es)
        ev = torch.cuda.Event()
        ev.record(side)
    main.wait_event(ev)
    for (plan, weights, _, _), e, Ho in zip(built, es, outs):
        plan.stage_b(e, weights, Ho)
    torch.cuda.synchronize()
    for Ho, Hr in zip(outs, ref):
        assert np.array_equal(bf16_bits(Ho), bf16_bits(Hr))


def test_argument_errors():
    w = BF16
    ids = W.token_stream(w)
    _, _, built = build(w, (1, 15), ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    plans = [b[0] for b in built]
    tables = [b[1].table for b in built]
    # another shape (row size) in the same launch
    w2 = w.scaled(row_dim=32)
    _, _, other = build(w2, (1,), ids.size)
    with pytest.raises(EngramError):
        stage_a_layers([plans[0], other[0][0]], ids_d, built[0][2], [tables[0], other[0][1].table])
    # tables in device and host memory mixed
    with pytest.raises(EngramError):
        stage_a_layers(plans, ids_d, built[0][2], [tables[0], tables[1].cpu().pin_memory()])
    # more layers than one launch takes
    with pytest.raises(EngramError):
        stage_a_layers(plans * 5, ids_d, built[0][2], tables * 5)
    with pytest.raises(ValueError):
        stage_a_layers(plans, ids_d, built[0][2], tables[:1])
    for p in plans:
        assert p.get_error() == (0, 0)


@pytest.mark.parametrize("N,K,row_dim,dtype,B,T", [
    (3, 8, 64, "i8", 3, 101),      # 16 rows of 64 bytes: 64 chunks, both halves full
    (4, 4, 32, "i8", 2, 77),       # 12 rows of 32 bytes: 24 chunks per token
    (3, 4, 16, "bf16", 5, 33),     # 8 rows of 32 bytes: 16 chunks
    (2, 3, 16, "f32", 1, 7),       # 3 rows of 64 bytes, 7 tokens: the last pair has one token
])
def test_half_warp_gather_shapes(N, K, row_dim, dtype, B, T):
    """Stage A where a token has at most 16 rows and 64 chunks (half a warp per
    token) against the oracle's gathered rows, odd token counts included, from
    HBM and from pinned host memory."""
    w = W.INT8_HOST.scaled(B=B, T=T, V=5000, V_proj=3850, prime_target=2003, d=256, span_copies=2, N=N, K=K,
                           row_dim=row_dim, table_dtype=dtype, act_dtype="f32" if dtype == "f32" else "bf16")
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, _ = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    z = O.hash_heads(O.project(ids, P), L.multipliers, L.primes, w.N, w.K, None)
    want = O.gather_concat(z.reshape(-1, w.R), L.tables(), w.table_dtype, L.table_scales())
    for host in (False, True):
        tab = to_torch(L.table, dtype, "cpu", pin=True) if host else weights.table
        e = plan.stage_a(ids_d, proj, tab, weights.scales)
        got = e.cpu().numpy() if dtype == "f32" else bf16_bits(e)
        exp = want.astype(np.float32) if dtype == "f32" else O.f64_to_bf16_bits(want)
        assert np.array_equal(got, exp.reshape(got.shape)), (dtype, host)
        assert plan.get_error() == (0, 0)
