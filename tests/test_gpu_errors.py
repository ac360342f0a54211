"""Host-made faults through the C ABI: every one is reported, none touches the GPU
outside what the kernels' own bounds checks allow.

Injected on the host: an index array with values past a table's row count
(the gather zero-fills those rows and flags ENGRAM_ERR_INDEX_RANGE), raw token
ids outside the vocabulary (clamped, flagged), pageable host tables
(ENGRAM_ERR_NOT_MAPPED before any launch), misaligned or null pointers and a
short workspace (refused before any launch)."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from hashed_gram_embedding_engram_gb300 import EngramError, _lib  # noqa: E402
from tests.gpu_helpers import bf16_bits, make_layer, to_torch  # noqa: E402

W_SMALL = W.PREFILL_BF16.scaled(B=2, T=100, V=5000, V_proj=3850, prime_target=4001, d=256)


@pytest.fixture(scope="module")
def layer():
    w = W_SMALL
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    return w, ids, P, L, plan, weights, proj, H


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_index_out_of_range_zero_fills_and_flags(layer):
    w, ids, P, L, plan, weights, proj, H = layer
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    assert plan.get_error() == (0, 0)
    bad = idx.clone()
    bad[5, 3] = int(L.primes[3])          # one past the last row of table 3
    bad[7, 0] = -1
    e = plan.gather(bad, weights.table)
    st, flags = plan.get_error()
    assert st == _lib.ERR_INDEX_RANGE and flags == 1
    assert plan.get_error() == (0, 0)     # reading clears the word
    rows = bf16_bits(e).reshape(-1, w.R, w.row_dim)
    assert np.all(rows[5, 3] == 0) and np.all(rows[7, 0] == 0)
    good = plan.gather(idx, weights.table)
    mask = np.ones(rows.shape[:2], bool)
    mask[5, 3] = mask[7, 0] = False
    assert np.array_equal(rows[mask], bf16_bits(good).reshape(-1, w.R, w.row_dim)[mask])


def test_raw_id_outside_vocabulary_is_flagged(layer):
    w, ids, P, L, plan, weights, proj, H = layer
    bad = torch.from_numpy(ids).cuda()
    bad[0, 3] = w.V + 10
    plan.hash(bad, proj)
    assert plan.get_error()[0] == _lib.ERR_INDEX_RANGE


def test_pageable_host_table_is_refused(layer):
    w, ids, P, L, plan, weights, proj, H = layer
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    e = torch.empty(idx.shape[0], w.d_mem, dtype=torch.bfloat16, device="cuda")
    pageable = np.ascontiguousarray(L.table)     # plain malloc'd host memory
    lib = _lib._lib()
    st = lib.engram_gather(plan._h, idx.data_ptr(), idx.shape[0], pageable.ctypes.data, None, e.data_ptr(),
                           stream())
    assert st == _lib.ERR_NOT_MAPPED
    with pytest.raises(ValueError):
        plan.gather(idx, torch.from_numpy(pageable.view(np.int16)).view(torch.bfloat16))


def test_misaligned_and_null_pointers_are_refused(layer):
    w, ids, P, L, plan, weights, proj, H = layer
    lib = _lib._lib()
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    e = torch.empty(idx.shape[0] * w.d_mem + 8, dtype=torch.bfloat16, device="cuda")
    st = lib.engram_gather(plan._h, idx.data_ptr(), idx.shape[0], weights.table.data_ptr(), None,
                           e.data_ptr() + 2, stream())
    assert st == _lib.ERR_INVALID_ARG
    st = lib.engram_gather(plan._h, None, idx.shape[0], weights.table.data_ptr(), None, e.data_ptr(), stream())
    assert st == _lib.ERR_INVALID_ARG
    st = lib.engram_hash(plan._h, None, 2, 100, proj.data_ptr(), w.V, None, idx.data_ptr(), stream())
    assert st == _lib.ERR_INVALID_ARG
    st = lib.engram_hash(plan._h, idx.data_ptr(), 2, 10 ** 6, proj.data_ptr(), w.V, None, idx.data_ptr(), stream())
    assert st == _lib.ERR_INVALID_ARG           # more tokens than the plan's max_tokens


def test_short_workspace_is_refused(layer):
    w, ids, P, L, plan, weights, proj, H = layer
    ws = torch.empty(plan.workspace_bytes(ids.size) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(EngramError) as ei:
        plan.forward(torch.from_numpy(ids).cuda(), proj, weights, H.clone(), workspace=ws)
    assert ei.value.status == _lib.ERR_WORKSPACE


def test_int8_table_without_scales_is_refused():
    w = W.INT8_HOST.scaled(B=1, T=50, V=5000, V_proj=3850, prime_target=3001, d=256, span_copies=1)
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    plan, weights, proj, H = make_layer(w, L, P, ids.size)
    idx = plan.hash(torch.from_numpy(ids).cuda(), proj)
    e = torch.empty(idx.shape[0], w.d_mem, dtype=torch.bfloat16, device="cuda")
    st = _lib._lib().engram_gather(plan._h, idx.data_ptr(), idx.shape[0], weights.table.data_ptr(), None,
                                   e.data_ptr(), stream())
    assert st == _lib.ERR_INVALID_ARG
    tab_host = to_torch(L.table, "i8", "cpu", pin=True)
    plan.gather(idx, tab_host, weights.scales)
    assert plan.get_error() == (0, 0)
