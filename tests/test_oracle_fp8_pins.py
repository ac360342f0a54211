"""Pins of the oracle's FP8 (e4m3) projection, CPU only.

What fixes them, independently of the oracle's code:
  * the e4m3 format itself (OCP 8-bit floating point, E4M3: bias 7, three
    mantissa bits, no infinities, largest finite 448, smallest subnormal
    2^-9): hand-picked values, ties and saturation;
  * torch's own float32 -> float8_e4m3fn conversion on every bf16 value in
    range (a library routine: round to nearest even);
  * exact cases: rows whose amax is 448 * 2^k and whose entries are e4m3 values
    times 2^k quantise without error, so the FP8 projection must equal the
    exact one; a planted dropped or swapped scale breaks that equality;
  * bounds: the codes are within half a grid step of x * 448/amax.
"""
import numpy as np
import pytest
import torch

from oracle import engram_oracle as O


@pytest.mark.parametrize("x,want", [
    (0.0, 0.0), (1.0, 1.0), (-1.0, -1.0), (448.0, 448.0), (-448.0, -448.0),
    (464.0, 448.0),              # above the largest finite value: saturates (480 would be NaN)
    (1e6, 448.0),
    (2.0 ** -9, 2.0 ** -9),      # smallest subnormal
    (2.0 ** -10, 0.0),           # half of it: tie, to the even neighbour 0
    (3 * 2.0 ** -10, 2.0 ** -8), # 1.5 subnormal steps: tie, to the even step count 2
    (2.0 ** -6, 2.0 ** -6),      # smallest normal
    (7 * 2.0 ** -9, 7 * 2.0 ** -9),  # largest subnormal
    (1.0625, 1.0),               # between 1 (m=0) and 1.125 (m=1): tie to even m
    (1.1875, 1.25),              # between 1.125 (m=1) and 1.25 (m=2): tie to even m
    (1.07, 1.125), (15.5, 16.0), (240.0, 240.0), (250.0, 256.0), (432.0, 448.0), (416.0, 416.0),
])
def test_e4m3_values_from_the_format(x, want):
    assert O.e4m3_round(np.float64(x)) == want
    assert O.e4m3_round(np.float64(-x)) == -want


def test_e4m3_matches_torch_conversion_on_every_bf16_in_range():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_matches_torch_on_random_float32():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * rng.choice([1e-3, 1e-1, 1, 30, 200], 200000)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(x.astype(np.float64)), ref)


def test_quantize_rows_codes_scales_and_bounds():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((6, 256)) * np.array([[1e-3], [0.02], [1], [5], [300], [1]])).astype(np.float32)
    x[5] = 0.0                                              # all-zero row
    q, s = O.quantize_rows_e4m3(x)
    assert s[5] == 1.0 and not q[5].any()
    for i in range(5):
        amax = np.float32(np.max(np.abs(x[i])))
        assert s[i] == np.float64(amax / np.float32(448))
        j = int(np.argmax(np.abs(x[i])))
        assert abs(q[i, j]) == 448.0                         # the row's extreme maps to the top code
        y = x[i].astype(np.float64) * np.float64(np.float32(448) / amax)
        a = np.abs(y)
        step = np.where(a >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3), 2.0 ** -9)
        assert np.all(np.abs(q[i] - y) <= 0.5 * step * (1 + 1e-6) + 1e-7 * a)


def test_quantize_rows_is_invariant_to_power_of_two_row_scaling():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    q, s = O.quantize_rows_e4m3(x)
    for k in (-7, -1, 3, 10):
        q2, s2 = O.quantize_rows_e4m3(x * np.float32(2.0 ** k))
        assert np.array_equal(q2, q) and np.array_equal(s2, s * 2.0 ** k)


def exact_fp8_operands(rng, rows, cols, exps):
    """Rows of e4m3 values times 2^k (k per row) whose amax is 448 * 2^k."""
    codes = O.e4m3_round(rng.standard_normal((rows, cols)) * 60)
    codes[:, 0] = 448.0 * np.where(rng.random(rows) < 0.5, 1, -1)
    return codes * (2.0 ** np.asarray(exps, dtype=np.float64))[:, None]


def test_fp8_projection_is_exact_on_exactly_representable_rows():
    rng = np.random.default_rng(11)
    d, M, dm = 16, 2, 64
    e = exact_fp8_operands(rng, 10, dm, rng.integers(-12, -4, 10))
    W = exact_fp8_operands(rng, (M + 1) * d, dm, rng.integers(-14, -6, (M + 1) * d))
    k8, v8 = O.kv_projection_fp8(e, W, d, M)
    k, v = O.kv_projection(e, W[:d], [W[(1 + m) * d:(2 + m) * d] for m in range(M)])
    assert np.array_equal(v8, v) and np.array_equal(k8, k)


def test_planted_scale_mistakes_are_caught():
    """A projection that drops the activation scale, or applies the weight
    scales by input instead of output row, disagrees with the exact product."""
    rng = np.random.default_rng(13)
    d, M, dm = 8, 1, 64
    e = exact_fp8_operands(rng, 6, dm, rng.integers(-12, -4, 6))
    W = exact_fp8_operands(rng, (M + 1) * d, dm, rng.integers(-14, -6, (M + 1) * d))
    exact = e @ W.T
    qe, se = O.quantize_rows_e4m3(e)
    qw, sw = O.quantize_rows_e4m3(W)
    assert np.array_equal((qe @ qw.T) * se[:, None] * sw, exact)
    assert not np.allclose((qe @ qw.T) * sw, exact)                       # activation scale dropped
    assert not np.allclose((qe @ qw.T) * se[:, None] * sw[::-1], exact)   # weight scales mis-assigned


def test_fp8_layer_stays_near_the_exact_layer():
    """On the tiny workload in bf16 form the FP8 forward is within the e4m3
    rounding (relative 2^-4 per operand) of the exact one, and not equal to it."""
    import workloads as W
    w = W.PREFILL_BF16.scaled(B=1, T=48, V=500, V_proj=385, prime_target=101, d=128)
    ids, P, L = W.token_stream(w), W.projection_map(w), W.layer_inputs(w, 1)
    ex = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype)
    f8 = O.forward(ids, P, L, w.N, w.K, w.conv_dil, w.eps, w.table_dtype, w.act_dtype, projection="fp8")
    for name in ("v", "k"):
        rel = np.linalg.norm(f8[name] - ex[name]) / np.linalg.norm(ex[name])
        assert 1e-4 < rel < 0.1, (name, rel)
    assert np.max(np.abs(f8["H_new"] - ex["H_new"])) < 0.5
