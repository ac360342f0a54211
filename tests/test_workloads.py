"""The seeded input generators: published test vectors and stated structure."""
import numpy as np

import workloads as W
from workloads import gen


def test_splitmix64_published_vectors():
    # reference outputs of splitmix64 (Steele, Lea & Flood 2014; Vigna's C version)
    assert W.splitmix64(0, 1) == [0xE220A8397B1DCDAF]
    assert W.splitmix64(1234567, 2) == [6457827717110365317, 3203168211198807973]


def test_multipliers_are_odd_and_ordered():
    m = W.hash_multipliers(W.TINY_F32, 0)
    assert m.dtype == np.uint64 and m.size == 2 * (2 + 3)
    assert np.all(m & np.uint64(1) == 1)
    assert [int(v) for v in m] == [v | 1 for v in W.splitmix64(1, 10)]
    m1 = W.hash_multipliers(W.PREFILL_BF16, 1)
    m15 = W.hash_multipliers(W.PREFILL_BF16, 15)
    assert m1.size == 8 * 5 and not np.array_equal(m1, m15)
    assert W.hash_multipliers(W.MULTIBRANCH_N4, 1).size == 8 * (2 + 3 + 4)


def test_primes_tiny_workload_match_stated_table_sizes():
    assert W.first_primes_from(1009, 4) == [1009, 1013, 1019, 1021]


def test_prime_totals_near_stated_row_counts():
    assert sum(W.first_primes_from(646400, 16)) == 10344164      # ~10342400 rows per layer
    assert abs(sum(W.first_primes_from(2500000, 16)) - 40_000_000) < 10_000
    assert abs(sum(W.first_primes_from(1500000, 24)) - 36_000_000) < 10_000


def test_projection_is_onto_and_many_to_one():
    for w in (W.TINY_F32, W.PREFILL_BF16):
        P = W.projection_map(w)
        assert P.shape == (w.V,) and P.min() >= 0 and P.max() < w.V_proj
        assert np.unique(P).size == w.V_proj
    assert round(0.77 * 129280) == W.PREFILL_BF16.V_proj


def test_token_stream_has_repeated_spans_and_zipf_head():
    w = W.PREFILL_BF16
    ids = W.token_stream(w)
    assert ids.shape == (1, 4096) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < w.V
    # the motif appears in span_copies aligned slots
    slots = ids[0].reshape(-1, w.span_len)
    _, counts = np.unique(slots, axis=0, return_counts=True)
    assert counts.max() >= w.span_copies
    # Zipf(1.1) over 129280: the top id takes several percent of tokens
    _, c = np.unique(ids, return_counts=True)
    assert c.max() / ids.size > 0.03


def test_int8_quantisation_recipe():
    q, s = gen.int8_rowscale_table(1000, 64, 0.02, 7, "t")
    assert q.dtype == np.int8 and s.dtype == np.float16
    assert np.abs(q.astype(int)).max() <= 127
    assert np.all(np.abs(q.astype(int)).max(axis=1) >= 120)      # each row uses its range
    x = q.astype(np.float64) * s.astype(np.float64)[:, None]
    assert abs(x.std() - 0.02) < 0.002


def test_layer_inputs_shapes_and_determinism():
    w = W.TINY_F32
    a = W.layer_inputs(w, 0)
    b = W.layer_inputs(w, 0)
    assert a.table.shape == (4062, 16) and a.table.dtype == np.float32
    assert a.W_kv.shape == (128, 64) and a.H.shape == (1, 64, 1, 64)
    assert a.row_offsets.tolist() == [0, 1009, 2022, 3041]
    for x, y in ((a.table, b.table), (a.W_kv, b.W_kv), (a.H, b.H), (a.conv, b.conv)):
        assert np.array_equal(x, y)
    assert [t.shape[0] for t in a.tables()] == [1009, 1013, 1019, 1021]
    assert abs(a.W_kv.std() - 0.125) < 0.01


def test_chunked_fill_independent_of_threads(monkeypatch):
    x1 = gen.normal_array((3, 1 << 23), 1.0, "bf16", 5, "k")
    monkeypatch.setattr(gen, "_threads", lambda: 1)
    x2 = gen.normal_array((3, 1 << 23), 1.0, "bf16", 5, "k")
    assert np.array_equal(x1, x2)
