"""Stage B as one cooperative launch -- the K/V projection and the conv linked
by per-row-block completion counters -- against the two-launch form (bit for
bit: the same tiles, the same operation order) and against the oracle.

The fused form applies to bf16 layers with one branch, w = 4 and d = 1024;
the cases vary the number and length of sequences (row blocks of 128 tokens
that straddle sequences, a ragged last block, two-position sequences) and the
dilation (its compile-time variants)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import engram_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from tests.gpu_helpers import act_to_f64, assert_close, make_layer  # noqa: E402

BASE = W.PREFILL_BF16.scaled(V=5000, V_proj=3850, prime_target=4001)


def layer(w):
    ids = W.token_stream(w)
    P = W.projection_map(w)
    L = W.layer_inputs(w, 1)
    return ids, P, L


def forward(w, ids, P, L, fused, timing=False, pairs=False):
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    plan.set_fused_stage_b(fused)
    plan.set_cta_pairs(pairs)
    if timing:
        plan.set_timing(True)
    plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H)
    n_kernels = len(plan.kernel_times()) if timing else None
    assert plan.get_error() == (0, 0)
    return H, n_kernels


def sample_positions(B, T):
    ts = sorted({0, 1, 2, 3, T // 2, T - 2, T - 1, min(127, T - 1), min(128, T - 1)} & set(range(T)))
    return [(b, t) for b in sorted({0, B - 1}) for t in ts]


# ordered by growing shared memory per block (longer tiles), so a launch that
# needs more than an earlier shape of the same dilation is covered
# (1, 2600, 3), (3, 900, 3), (1, 4096, 3) and (16, 2048, 3) give the two-launch form's
# projection 256-column tiles, which can also run on CTA pairs (gemm_pair.cu);
# 2600 and 2700 rows leave a ragged last pair tile whose second CTA holds no
# valid row.  The pair form is compared with the same bits.
@pytest.mark.parametrize("B,T,dil", [(5, 2, 3), (7, 37, 5), (2, 129, 1), (3, 700, 3), (1, 1000, 8), (1, 2600, 3),
                                     (3, 900, 3), (1, 4096, 3), (16, 2048, 3)])
def test_fused_stage_b_equals_two_launches_and_oracle(B, T, dil):
    w = BASE.scaled(B=B, T=T, conv_dil=dil)
    ids, P, L = layer(w)
    H_fused, n_fused = forward(w, ids, P, L, True, timing=True)
    H_split, n_split = forward(w, ids, P, L, False, timing=True)
    H_pairs, n_pairs = forward(w, ids, P, L, False, timing=True, pairs=True)
    assert n_pairs == n_split
    assert torch.equal(H_pairs.view(torch.int16), H_split.view(torch.int16))
    # the fused form ran: one traced interval for Stage B; the two-launch form
    # has two, or three with the finalize kernel where its projection tiles are
    # narrower than 256 columns (fewer than one tile of that width per SM)
    assert n_fused == 2 and n_split in (3, 4)
    assert torch.equal(H_fused.view(torch.int16), H_split.view(torch.int16))
    if B * T <= 300:
        ref = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)["H_new"]
        assert_close(act_to_f64(H_fused), ref, "bf16", "fused")
    else:
        pos = sample_positions(B, T)
        ref = O.forward_at(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, pos)
        got = np.stack([act_to_f64(H_fused[b, t]) for b, t in pos])
        assert_close(got, ref, "bf16", "fused sampled")


def test_fused_stage_b_streams_chunks_bit_identically():
    """Chunks of 300 positions with the streaming state (the fused launch, then
    the state update) reproduce one-shot prefill by the two-launch form."""
    from hashed_gram_embedding_engram_gb300 import EngramState
    w = BASE.scaled(B=2, T=1100)
    ids, P, L = layer(w)
    full, _ = forward(w, ids, P, L, False)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    plan.set_fused_stage_b(True)
    st = EngramState.zeros(plan, w.B)
    ids_d = torch.from_numpy(ids).cuda()
    out = H.clone()
    for t0 in range(0, w.T, 300):
        t1 = min(t0 + 300, w.T)
        seg = out[:, t0:t1].contiguous()
        plan.forward(ids_d[:, t0:t1].contiguous(), proj, weights, seg, st)
        out[:, t0:t1] = seg
    assert plan.get_error() == (0, 0)
    assert torch.equal(st.pos.cpu(), torch.full((w.B,), w.T, dtype=torch.int32))
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))


def test_fused_stage_b_repeats_and_reuses_its_workspace():
    """The counters in the workspace are zeroed by every call: repeated calls on
    one workspace, in a CUDA graph and eagerly, give the same bits."""
    w = BASE.scaled(B=2, T=900)
    ids, P, L = layer(w)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    ws = plan.new_workspace(ids.size)
    ref = H0.clone()
    plan.forward(ids_d, proj, weights, ref, None, ws)
    H = H0.clone()
    for _ in range(3):
        H.copy_(H0)
        plan.forward(ids_d, proj, weights, H, None, ws)
        assert torch.equal(H.view(torch.int16), ref.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            plan.forward(ids_d, proj, weights, H, None, ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        H.copy_(H0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(H.view(torch.int16), ref.view(torch.int16))
    assert plan.get_error() == (0, 0)


def test_tracing_inside_a_graph():
    """A traced call captured into a CUDA graph records its events as graph
    nodes: every replay gives one interval per kernel, and the same bits."""
    w = BASE.scaled(B=2, T=900)
    ids, P, L = layer(w)
    ref, _ = forward(w, ids, P, L, False)
    plan, weights, proj, H0 = make_layer(w, L, P, ids.size)
    ids_d = torch.from_numpy(ids).cuda()
    ws = plan.new_workspace(ids.size)
    H = H0.clone()
    plan.set_timing(True)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            plan.forward(ids_d, proj, weights, H, None, ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        H.copy_(H0)
        g.replay()
        torch.cuda.synchronize()
        t = plan.kernel_times()
        assert len(t) in (3, 4) and all(x > 0 for x in t)
        assert torch.equal(H.view(torch.int16), ref.view(torch.int16))
    assert plan.get_error() == (0, 0)
