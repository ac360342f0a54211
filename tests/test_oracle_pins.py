"""Pins of the CPU oracle against facts the pages and mathematics fix.

Nothing here compares the oracle with itself: each check is a hand-worked value,
a closed form, an invariant the pages state, a library routine that computes
the same special case, or a brute-force re-evaluation along another route.
Page cited throughout: "DeepSeek Engram 系列导读" (foosynaptic.github.io),
section "Engram 工作原理", Steps 1-8, and "多分支 backbone 上的变体".
"""
import math
import os
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from oracle import engram_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- #
# helpers: tiny hand-built layers
# --------------------------------------------------------------------------- #
def tiny_layer(rng, N=3, K=2, row=4, d=8, M=1, w=4, primes=(1009, 1013, 1019, 1021, 1031, 1033),
               B=2, T=24, mults=None, table_scale=0.5):
    R = (N - 1) * K
    primes = np.array(primes[:R], dtype=np.uint32)
    offs = np.zeros(R, dtype=np.int64)
    offs[1:] = np.cumsum(primes.astype(np.int64))[:-1]
    rows = int(primes.sum())
    if mults is None:
        mults = (rng.integers(0, 2**63, size=sum(K * n for n in range(2, N + 1)), dtype=np.uint64) * np.uint64(2)
                 + np.uint64(1))
    L = SimpleNamespace(
        multipliers=np.asarray(mults, dtype=np.uint64), primes=primes, row_offsets=offs,
        table=(table_scale * rng.standard_normal((rows, row))).astype(np.float32), scales=None,
        W_kv=(rng.standard_normal(((M + 1) * d, R * row)) / math.sqrt(R * row)).astype(np.float32),
        g_h=(1 + 0.1 * rng.standard_normal((M, d))).astype(np.float32),
        g_k=(1 + 0.1 * rng.standard_normal((M, d))).astype(np.float32),
        g_c=(1 + 0.1 * rng.standard_normal(d)).astype(np.float32),
        conv=(0.5 * rng.standard_normal((d, w))).astype(np.float32),
        H=rng.standard_normal((B, T, M, d)).astype(np.float32),
    )
    L.tables = lambda: [L.table[o:o + int(p)] for o, p in zip(L.row_offsets, L.primes)]
    L.table_scales = lambda: None
    return L


def run(ids, P, L, N=3, K=2, dil=3, eps=1e-6, state=None):
    return O.forward(ids, P, L, N, K, dil, eps, "f32", "f32", state)


# --------------------------------------------------------------------------- #
# Steps 2-3: hand-worked hash values
# --------------------------------------------------------------------------- #
# multipliers in flat order (n, k, i): n=2: k=0 -> 3, 5; k=1 -> 7, 11
#                                      n=3: k=0 -> 13, 17, 19; k=1 -> 23, 29, 31
HAND_MULTS = np.array([3, 5, 7, 11, 13, 17, 19, 23, 29, 31], dtype=np.uint64)
HAND_PRIMES = [1009, 1013, 1019, 1021]


def test_hash_hand_worked_small_values():
    xp = np.array([[4, 9, 2]], dtype=np.int64)
    z = O.hash_heads(xp, HAND_MULTS, HAND_PRIMES, N=3, K=2)
    # t=0: window (x'_0, pad, pad) = (4, 0, 0)
    #   (2,0): 4*3 ^ 0*5 = 12            (2,1): 4*7 = 28
    #   (3,0): 4*13 = 52                 (3,1): 4*23 = 92
    assert z[0, 0].tolist() == [12, 28, 52, 92]
    # t=1: (x'_1, x'_0, pad) = (9, 4, 0)
    #   (2,0): 27 ^ 20 = 0b11011 ^ 0b10100 = 0b01111 = 15
    #   (2,1): 63 ^ 44 = 0b111111 ^ 0b101100 = 0b010011 = 19
    #   (3,0): 117 ^ 68 ^ 0 = 0b1110101 ^ 0b1000100 = 0b0110001 = 49
    #   (3,1): 207 ^ 116 = 0b11001111 ^ 0b01110100 = 0b10111011 = 187
    assert z[0, 1].tolist() == [15, 19, 49, 187]
    # t=2: (x'_2, x'_1, x'_0) = (2, 9, 4)
    #   (2,0): 6 ^ 45 = 0b000110 ^ 0b101101 = 0b101011 = 43
    #   (2,1): 14 ^ 99 = 0b0001110 ^ 0b1100011 = 0b1101101 = 109
    #   (3,0): 26 ^ 153 ^ 76 = 0b00011010 ^ 0b10011001 ^ 0b01001100 = 0b11001111 = 207
    #   (3,1): 46 ^ 261 ^ 124 = 0b000101110 ^ 0b100000101 ^ 0b001111100 = 0b101010111 = 343
    assert z[0, 2].tolist() == [43, 109, 207, 343]


def test_hash_reduces_modulo_prime():
    # x'=100, m(2,0,0)=3 -> 300 < 1009 stays; a value above p wraps: 97*13 = 1261 -> 1261-1019 = 242
    xp = np.array([[97]], dtype=np.int64)
    z = O.hash_heads(xp, HAND_MULTS, HAND_PRIMES, N=3, K=2)
    # (2,0): 291; (2,1): 679; (3,0): 1261 mod 1019 = 242; (3,1): 2231 mod 1021 = 2231-2042 = 189
    assert z[0, 0].tolist() == [291, 679, 242, 189]


def test_hash_wraps_modulo_2_64():
    # m = 2^63 + 1.  x * m = x*2^63 + x: for x = 3 that is 2^64 + 2^63 + 3 == 2^63 + 3 (mod 2^64);
    # for x = 6 it is 3*2^64 + 6 == 6.  A signed or floating product would differ.
    big = (1 << 63) + 1
    mults = np.array([big, 1, big, 1, big, 1, 1, big, 1, 1], dtype=np.uint64)
    for x, low in ((3, (1 << 63) + 3), (6, 6)):
        xp = np.array([[x]], dtype=np.int64)
        z = O.hash_heads(xp, mults, HAND_PRIMES, N=3, K=2)
        expect = [low % p for p in HAND_PRIMES]          # Python big ints, exact
        # closed form for 2^63 + 3 by modular exponentiation, a separate route
        if x == 3:
            assert expect == [(pow(2, 63, p) + 3) % p for p in HAND_PRIMES]
        assert z[0, 0].tolist() == expect


def test_hash_uses_prev_ids_for_window_before_start():
    # continuing a sequence: x'_{-2}, x'_{-1} = 4, 9 and then x'_0 = 2 must hash like t=2 above
    xp = np.array([[2]], dtype=np.int64)
    prev = np.array([[4, 9]], dtype=np.int64)
    z = O.hash_heads(xp, HAND_MULTS, HAND_PRIMES, N=3, K=2, prev=prev)
    assert z[0, 0].tolist() == [43, 109, 207, 343]


def test_suffix_ngram_matches_page_example():
    rows = []
    with open(os.path.join(GOLDEN, "ngram_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            sent, pos, n, expect = [s.strip() for s in line.split("|")]
            rows.append((sent.split(), int(pos), int(n), expect.split()))
    assert rows
    for words, pos, n, expect in rows:
        vocab = {wd: i + 1 for i, wd in enumerate(dict.fromkeys(words))}
        inv = {i: wd for wd, i in vocab.items()}
        xp = np.array([[vocab[wd] for wd in words]], dtype=np.int64)
        win = O.suffix_ngram(xp, n)                      # [x'_t, x'_{t-1}, ...]
        got = [inv[int(win[i][0, pos])] for i in reversed(range(n))]
        assert got == expect


def test_shared_suffix_shares_lower_order_indices():
    # "Peter the Great" and "Alexander the Great": same 2-gram at "Great", different 3-gram
    rng = np.random.default_rng(3)
    mults = rng.integers(0, 2**63, size=10, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    PETER, ALEX, THE, GREAT = 11, 12, 13, 14
    xp = np.array([[PETER, THE, GREAT, ALEX, THE, GREAT]], dtype=np.int64)
    z = O.hash_heads(xp, mults, HAND_PRIMES, N=3, K=2)
    assert z[0, 2, :2].tolist() == z[0, 5, :2].tolist()   # order 2, both heads
    assert z[0, 2, 2:].tolist() != z[0, 5, 2:].tolist()   # order 3 differs


def test_projection_merges_ids():
    # Step 1: two raw ids with one canonical id get identical indices (Apple / " apple")
    P = np.array([0, 5, 7, 5, 9], dtype=np.int64)      # raw 1 and 3 -> 5
    rng = np.random.default_rng(0)
    mults = rng.integers(0, 2**63, size=10, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    a = O.hash_heads(O.project(np.array([[2, 1]]), P), mults, HAND_PRIMES, 3, 2)
    b = O.hash_heads(O.project(np.array([[2, 3]]), P), mults, HAND_PRIMES, 3, 2)
    assert np.array_equal(a, b)


def test_indices_depend_only_on_suffix_window():
    rng = np.random.default_rng(1)
    mults = rng.integers(0, 2**63, size=10, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    xp = rng.integers(0, 700, size=(1, 20))
    z = O.hash_heads(xp, mults, HAND_PRIMES, 3, 2)
    t = 12
    for n in (2, 3):
        cols = slice((n - 2) * 2, (n - 1) * 2)
        far = xp.copy()
        far[0, t - n] += 1                                # just outside the n-gram
        assert np.array_equal(O.hash_heads(far, mults, HAND_PRIMES, 3, 2)[0, t, cols], z[0, t, cols])
        near = xp.copy()
        near[0, t - n + 1] += 1                           # oldest id inside the n-gram
        assert not np.array_equal(O.hash_heads(near, mults, HAND_PRIMES, 3, 2)[0, t, cols], z[0, t, cols])
    later = xp.copy()
    later[0, t + 1:] += 1
    assert np.array_equal(O.hash_heads(later, mults, HAND_PRIMES, 3, 2)[0, :t + 1], z[0, :t + 1])


def test_windows_do_not_cross_sequences():
    rng = np.random.default_rng(2)
    mults = rng.integers(0, 2**63, size=10, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    xp = rng.integers(1, 700, size=(2, 5))
    z = O.hash_heads(xp, mults, HAND_PRIMES, 3, 2)
    alone = O.hash_heads(xp[1:], mults, HAND_PRIMES, 3, 2)
    assert np.array_equal(z[1], alone[0])


# --------------------------------------------------------------------------- #
# Step 4: gather + concat, dequant
# --------------------------------------------------------------------------- #
def test_gather_concat_brute_force():
    rng = np.random.default_rng(4)
    tabs = [rng.standard_normal((p, 3)).astype(np.float32) for p in (7, 11, 13, 17)]
    z = np.stack([rng.integers(0, p, size=(2, 5)) for p in (7, 11, 13, 17)], axis=-1)
    e = O.gather_concat(z, tabs, "f32")
    for b in range(2):
        for t in range(5):
            expect = []
            for r in range(4):                            # n-major, then k
                expect.extend(float(v) for v in tabs[r][z[b, t, r]])
            assert e[b, t].tolist() == expect


def test_bf16_widening_and_rounding_agree_with_torch():
    rng = np.random.default_rng(5)
    x32 = (rng.standard_normal(4096) * 0.02).astype(np.float32)
    bits_torch = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16_bits(x32.astype(np.float64)), bits_torch)
    widened_torch = torch.from_numpy(bits_torch.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_to_f64(bits_torch), widened_torch)
    # ties go to even: 1 + 2^-8 is halfway between bf16 1 and 1 + 2^-7
    assert O.f64_to_bf16_bits(np.array([1 + 2.0 ** -8]))[0] == 0x3F80
    assert O.f64_to_bf16_bits(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82


def test_int8_dequant_is_one_bf16_rounding_of_the_exact_product():
    rng = np.random.default_rng(18)
    q = rng.integers(-127, 128, size=(50, 64)).astype(np.int8)
    s = (rng.random(50) * 1e-3 + 1e-4).astype(np.float16)
    e = O.gather_concat(np.arange(50)[:, None], [q], "i8", [s])
    # int8 (8 bits) times fp16 (11 bits) fits binary32's 24 bits: the product is exact there
    prod32 = torch.from_numpy(q.astype(np.float32)) * torch.from_numpy(s.astype(np.float32))[:, None]
    assert np.array_equal(prod32.double().numpy(), q.astype(np.float64) * s.astype(np.float64)[:, None])
    # and the row the gather produces is torch's bf16 rounding of it
    assert np.array_equal(e, prod32.to(torch.bfloat16).double().numpy())
    assert e[0, 0] == O.bf16_to_f64(O.f64_to_bf16_bits(np.array([float(q[0, 0]) * float(s[0])])))[0]


# --------------------------------------------------------------------------- #
# Steps 5-6: projection and gate
# --------------------------------------------------------------------------- #
def test_kv_projection_against_python_loops():
    rng = np.random.default_rng(6)
    e = rng.standard_normal((3, 6))
    WV = rng.standard_normal((4, 6))
    WK = [rng.standard_normal((4, 6)) for _ in range(2)]
    k, v = O.kv_projection(e, WV, WK)
    for t in range(3):
        for c in range(4):
            assert v[t, c] == pytest.approx(sum(WV[c, j] * e[t, j] for j in range(6)), rel=1e-13)
            for m in range(2):
                assert k[t, m, c] == pytest.approx(sum(WK[m][c, j] * e[t, j] for j in range(6)), rel=1e-13)


def test_rmsnorm_closed_form():
    y = O.rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert y.tolist() == pytest.approx([3 / r, 8 / r], rel=1e-15)


def test_gate_hand_worked():
    # h = (1, 3), k = (2, -1), unit weights, eps = 0:
    # rms(h) = sqrt(5), rms(k) = sqrt(2.5), <h,k>/(rms rms) = -1/sqrt(12.5); / sqrt(2) = -1/5
    a = O.gate(np.array([[1.0, 3.0]]), np.array([[2.0, -1.0]]), np.ones((1, 2)), np.ones((1, 2)), 0.0)
    assert a[0] == pytest.approx(1 / (1 + math.exp(0.2)), rel=1e-15)


def test_gate_aligned_and_opposed_closed_form():
    rng = np.random.default_rng(7)
    d = 64
    h = rng.standard_normal((1, d))
    g = np.ones((1, d))
    a_same = O.gate(h, h, g, g, 0.0)[0]
    a_opp = O.gate(h, -h, g, g, 0.0)[0]
    # <x/rms, x/rms> = d, so the logit is d / sqrt(d) = sqrt(d)
    assert a_same == pytest.approx(1 / (1 + math.exp(-math.sqrt(d))), rel=1e-14)
    assert a_opp == pytest.approx(1 / (1 + math.exp(math.sqrt(d))), rel=1e-12)
    assert 0.0 < a_opp < 0.5 < a_same < 1.0


def test_gate_in_open_unit_interval_on_workload_scale():
    rng = np.random.default_rng(8)
    M, d = 4, 256
    h = rng.standard_normal((500, M, d))
    k = 0.02 * rng.standard_normal((500, M, d))
    g = 1 + 0.1 * rng.standard_normal((M, d))
    a = O.gate(h, k, g, g, 1e-6)
    assert a.shape == (500, M)
    assert np.all(a > 0) and np.all(a < 1)


# --------------------------------------------------------------------------- #
# Step 7: convolution
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("w,dil", [(4, 3), (4, 4), (3, 2)])
def test_conv_matches_torch_depthwise_conv1d(w, dil):
    rng = np.random.default_rng(9)
    B, T, d = 2, 30, 5
    u = rng.standard_normal((B, T, d))
    conv = rng.standard_normal((d, w))
    got = O.dilated_causal_conv(u, conv, dil)
    x = torch.from_numpy(u).permute(0, 2, 1)                       # [B, d, T]
    x = torch.nn.functional.pad(x, ((w - 1) * dil, 0))             # causal: left zeros
    ref = torch.nn.functional.conv1d(x, torch.from_numpy(conv)[:, None, :], groups=d, dilation=dil)
    assert np.allclose(got, ref.permute(0, 2, 1).numpy(), rtol=1e-13, atol=1e-13)


def test_conv_branch_lag0_only_closed_form():
    rng = np.random.default_rng(10)
    vt = 0.01 * rng.standard_normal((1, 9, 6))
    gc = 1 + 0.1 * rng.standard_normal(6)
    c = rng.standard_normal(6)
    conv = np.zeros((6, 4))
    conv[:, 3] = c                                                  # tap w-1 = lag 0
    Y = O.conv_branch(vt, gc, conv, 3, 1e-6)
    u = vt / np.sqrt(np.mean(vt * vt, axis=-1, keepdims=True) + 1e-6) * gc
    x = torch.from_numpy(c * u)
    assert np.allclose(Y, torch.nn.functional.silu(x).numpy() + vt, rtol=1e-13, atol=1e-15)


def test_receptive_field_is_one_plus_w_minus_1_times_N():
    # w = 4, dilation N = 3: Y_t reads vt_{t-9} but not vt_{t-10}; 1 + (w-1)N = 10 positions
    rng = np.random.default_rng(11)
    T, d, t = 30, 4, 25
    vt = rng.standard_normal((1, T, d))
    gc = np.ones(d)
    conv = rng.standard_normal((d, 4))
    base = O.conv_branch(vt, gc, conv, 3, 1e-6)[0, t]
    seen = []
    for lag in range(0, 12):
        p = vt.copy()
        p[0, t - lag] *= 3.0
        p[0, t - lag, 0] += 1.0
        seen.append(not np.array_equal(O.conv_branch(p, gc, conv, 3, 1e-6)[0, t], base))
    assert [lag for lag, s in enumerate(seen) if s] == [0, 3, 6, 9]
    assert max(lag for lag, s in enumerate(seen) if s) + 1 == 1 + (4 - 1) * 3


# --------------------------------------------------------------------------- #
# the whole layer
# --------------------------------------------------------------------------- #
def test_zero_table_leaves_H_unchanged():
    rng = np.random.default_rng(12)
    L = tiny_layer(rng)
    L.table[:] = 0
    ids = rng.integers(0, 50, size=(2, 24))
    P = rng.integers(0, 40, size=50)
    out = run(ids, P, L)
    assert np.all(out["alpha"] == 0.5)                    # sigma(0)
    assert np.array_equal(out["H_new"], L.H.astype(np.float64))


def test_identity_projection_no_conv_gives_alpha_times_e():
    # d_mem = d, W_V = I, conv = 0: SiLU(0) = 0, so Y = alpha * e and H_new = H + alpha e
    rng = np.random.default_rng(13)
    L = tiny_layer(rng, row=2, d=8)                        # R = 4 rows of 2 -> d_mem = 8 = d
    L.W_kv[:8] = np.eye(8, dtype=np.float32)
    L.conv[:] = 0
    ids = rng.integers(0, 50, size=(2, 24))
    P = rng.integers(0, 40, size=50)
    out = run(ids, P, L)
    expect = L.H.astype(np.float64) + out["alpha"][..., None] * out["e"][:, :, None, :]
    assert np.allclose(out["H_new"], expect, rtol=1e-14, atol=1e-15)


def test_layer_causality_and_token_receptive_field():
    # Y_t depends on raw tokens t-11 .. t (hash reach N-1 = 2, conv reach (w-1)N = 9)
    rng = np.random.default_rng(14)
    L = tiny_layer(rng, B=1, T=40)
    ids = rng.integers(0, 50, size=(1, 40))
    P = np.arange(50)
    base = run(ids, P, L)["H_new"]
    t = 30
    for tp in range(40):
        p = ids.copy()
        p[0, tp] = (p[0, tp] + 17) % 50
        changed = not np.array_equal(run(p, P, L)["H_new"][0, t], base[0, t])
        assert changed == (t - 11 <= tp <= t), tp
    # h after t does not reach t either
    L2 = tiny_layer(np.random.default_rng(14), B=1, T=40)
    L2.H[0, t + 1:] += 1.0
    assert np.array_equal(run(ids, P, L2)["H_new"][0, :t + 1], base[0, :t + 1])


def test_windowed_evaluation_matches_full_sequence():
    rng = np.random.default_rng(15)
    L = tiny_layer(rng, B=2, T=24)
    ids = rng.integers(0, 50, size=(2, 24))
    P = rng.integers(0, 40, size=50)
    full = run(ids, P, L)["H_new"]
    pos = [(b, t) for b in range(2) for t in range(24)]
    win = O.forward_at(ids, P, L, 3, 2, 3, 1e-6, "f32", "f32", pos)
    assert np.allclose(win, np.stack([full[b, t] for b, t in pos]), rtol=1e-12, atol=1e-12)


def test_decode_steps_equal_prefill():
    rng = np.random.default_rng(16)
    L = tiny_layer(rng, B=3, T=20)
    ids = rng.integers(0, 50, size=(3, 20))
    P = rng.integers(0, 40, size=50)
    full = run(ids, P, L)["H_new"]
    Lp = tiny_layer(np.random.default_rng(16), B=3, T=20)
    Lp.H = L.H[:, :13].copy()
    st = run(ids[:, :13], P, Lp)["state"]
    for t in range(13, 20):
        Lt = tiny_layer(np.random.default_rng(16), B=3, T=20)
        Lt.H = L.H[:, t:t + 1].copy()
        o = run(ids[:, t:t + 1], P, Lt, state=st)
        st = o["state"]
        assert np.allclose(o["H_new"][:, 0], full[:, t], rtol=1e-12, atol=1e-12)


def test_multibranch_one_branch_and_permutation():
    rng = np.random.default_rng(17)
    L = tiny_layer(rng, M=3, d=8, B=1, T=16)
    ids = rng.integers(0, 50, size=(1, 16))
    P = rng.integers(0, 40, size=50)
    out = run(ids, P, L)["H_new"]
    # branch m alone, as a one-branch layer with W_K^(m), h^(m), gate weights m
    for m in range(3):
        Lm = tiny_layer(np.random.default_rng(17), M=3, d=8, B=1, T=16)
        Lm.W_kv = np.concatenate([L.W_kv[:8], L.W_kv[(1 + m) * 8:(2 + m) * 8]])
        Lm.g_h, Lm.g_k = L.g_h[m:m + 1], L.g_k[m:m + 1]
        Lm.H = L.H[:, :, m:m + 1]
        assert np.allclose(run(ids, P, Lm)["H_new"][:, :, 0], out[:, :, m], rtol=1e-13, atol=1e-13)
    # permuting branches (h, W_K, gate weights together) permutes outputs
    perm = [2, 0, 1]
    Lq = tiny_layer(np.random.default_rng(17), M=3, d=8, B=1, T=16)
    Lq.W_kv = np.concatenate([L.W_kv[:8]] + [L.W_kv[(1 + m) * 8:(2 + m) * 8] for m in perm])
    Lq.g_h, Lq.g_k, Lq.H = L.g_h[perm], L.g_k[perm], L.H[:, :, perm]
    assert np.allclose(run(ids, P, Lq)["H_new"], out[:, :, perm], rtol=1e-13, atol=1e-13)
