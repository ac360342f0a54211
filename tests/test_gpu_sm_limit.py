"""Stage B's persistent kernels limited to fewer SMs (engram_plan_set_sm_limit)
give the same bits as on all SMs, and a batch in pieces -- each piece's Stage A
over host-memory tables on a side stream, beside the previous piece's Stage B
limited to the SMs the lookup leaves free -- equals one call."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from tests.gpu_helpers import make_layer, to_torch  # noqa: E402

BF16 = W.PREFILL_BF16.scaled(V=5000, V_proj=3850, prime_target=4001)
I8 = W.INT8_HOST.scaled(B=8, T=600, V=5000, V_proj=3850, prime_target=3001, span_copies=3)


def bits(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("B,T,limit", [(1, 4096, 114), (2, 1300, 37), (3, 500, 1), (1, 2600, 0)])
def test_sm_limit_keeps_the_bits(B, T, limit):
    w = BF16.scaled(B=B, T=T)
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    ref = H0.clone()
    plan.forward(ids_d, proj, weights, ref)
    plan.set_sm_limit(limit)
    got = H0.clone()
    plan.forward(ids_d, proj, weights, got)
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(got), bits(ref))


def test_pieces_beside_a_host_table_lookup_equal_one_call():
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
    assert 0 < plan.host_gather_sms() < torch.cuda.get_device_properties(0).multi_processor_count
    plan.set_sm_limit(torch.cuda.get_device_properties(0).multi_processor_count - plan.host_gather_sms())
    pieces = [(0, 3), (3, 5), (5, 8)]
    es = [torch.empty((hi - lo) * w.T, w.d_mem, dtype=torch.bfloat16, device="cuda") for lo, hi in pieces]
    H = H0.clone()
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    side.wait_stream(main)
    ready = []
    with torch.cuda.stream(side):
        for (lo, hi), ep in zip(pieces, es):
            plan.stage_a(ids_d[lo:hi], proj, table_host, weights.scales, out=ep)
            ev = torch.cuda.Event()
            ev.record(side)
            ready.append(ev)
    for (lo, hi), ep, ev in zip(pieces, es, ready):
        main.wait_event(ev)
        plan.stage_b(ep, weights, H[lo:hi])
    torch.cuda.synchronize()
    assert plan.get_error() == (0, 0)
    assert torch.equal(bits(H), bits(ref))
