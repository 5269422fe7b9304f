"""Pins of the CPU oracle to facts outside itself (CPU only).

Each pin is chosen so that a plausible mistake in the oracle (nibble order,
zero point, scale index, a transposed operand, a dropped term, a sign) fails
at least one of them; ``test_mutants_are_caught`` plants such mistakes in the
oracle (compile-time mutants, CPU only) and checks that they are caught.
"""
from fractions import Fraction
import math
import os

import numpy as np
import pytest

import oracle as oracle_mod
from int4_weight_only_q4f16_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Pack codes [N, K] (0..15) into words [N, K/8], element i of a word in
    bits 4i..4i+3 (the packing the docs page's extraction rule inverts)."""
    N, K = codes.shape
    c = codes.reshape(N, K // 8, 8).astype(np.uint64)
    words = np.zeros((N, K // 8), dtype=np.uint64)
    for i in range(8):
        words |= c[:, :, i] << np.uint64(4 * i)
    return words.astype(np.uint32)


def codes_by_hex(word: int):
    """Independent route to a word's codes: its 8-digit hex string read from
    the right (element 0 is the last hex digit)."""
    s = "%08x" % (word & 0xFFFFFFFF)
    return [int(s[7 - i], 16) for i in range(8)]


# --------------------------------------------------------------------------
# binary16 conversions against numpy's (a library routine)
# --------------------------------------------------------------------------
def test_f16_decode_all_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle.f16_to_f64(0x8000)) == -1.0


def test_f16_encode_round_to_nearest_even(oracle):
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact ties between adjacent f16 values, normal and subnormal
        (np.arange(1024, 1100) + 0.5) * 2.0 ** -10,
        (np.arange(0, 60) + 0.5) * 2.0 ** -24,
        [65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -26, -2.0 ** -25,
         3 * 2.0 ** -26, 0.0, -0.0, 6.1e-5, 2.0 ** -14 - 2.0 ** -25],
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16)
    got = oracle.round_f16(vals)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_tolerance_admits_correctly_rounded_f16_outputs():
    """The outputs are f16, so the parity bar must admit f16_rn(y_ref) for
    every y_ref in f16 range, normal or subnormal, even with S = 0 (numpy's
    f16 conversion as the rounding)."""
    rng = np.random.default_rng(11)
    y = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-12, 4, 20000),
                        (np.arange(0, 200) + 0.5) * 2.0 ** -24, [0.0, 2.0 ** -25, 6.5e4]])
    err = np.abs(y.astype(np.float16).astype(np.float64) - y)
    assert np.all(err <= oracle_mod.tolerance(y, np.zeros_like(y)))
    # and the absolute term is no larger than it must be: half the f16
    # subnormal spacing, attained at an exact tie
    t = 2.0 ** -25
    assert oracle_mod.tolerance(0.0, 0.0) == t


# --------------------------------------------------------------------------
# the format, from the golden fixtures
# --------------------------------------------------------------------------
def test_nibble_order_golden(oracle):
    for row in _rows("nibble_order.txt"):
        word = int(row[0], 16)
        want = [int(v) for v in row[1:]]
        wq = np.array([[word]], dtype=np.uint32)
        got = [oracle.code(wq, 8, 0, k) for k in range(8)]
        assert got == want, hex(word)
        assert codes_by_hex(word) == want


def test_dequant_golden(oracle):
    for code, sbits, sdec, want in _rows("dequant_values.txt"):
        code, sbits = int(code), int(sbits, 16)
        assert oracle.f16_to_f64(sbits) == float(sdec)
        K = 32
        wq = pack_codes(np.full((1, K), code, dtype=np.int64))
        sc = np.array([[sbits]], dtype=np.uint16).view(np.float16)
        w = oracle.dequant(wq, sc, 1, K)
        assert np.all(w == float(want)), (code, hex(sbits))


def test_pack_unpack_round_trip(oracle):
    rng = np.random.default_rng(1)
    N, K = 5, 96
    codes = rng.integers(0, 16, (N, K))
    wq = pack_codes(codes)
    for n in range(N):
        for k in range(K):
            assert oracle.code(wq, K, n, k) == codes[n, k]
    # and the independent hex-digit route agrees with the packing
    for n in range(N):
        flat = sum((codes_by_hex(int(w)) for w in wq[n]), [])
        assert flat == list(codes[n])


# --------------------------------------------------------------------------
# GEMV: one-hot columns, closed form, brute force, linearity
# --------------------------------------------------------------------------
def _patterned(N, K, seed=3):
    """codes q[n,k] = (n + 3k) mod 16 and distinct scales per (n, group)."""
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    codes = (n + 3 * k) % 16
    rng = np.random.default_rng(seed)
    sc = (rng.random((N, K // 32)) * 0.9 + 0.05).astype(np.float16)
    return codes, pack_codes(codes), sc


def test_one_hot_columns_exact(oracle):
    """x = e_k must return exactly column k of the dequantized matrix; N != K
    so that a transposed operand cannot pass."""
    N, K = 12, 96
    codes, wq, sc = _patterned(N, K)
    for k in range(K):
        x = np.zeros((1, K), dtype=np.float16)
        x[0, k] = 1.0
        y, S = oracle.gemv(wq, sc, x, N, K)
        want = (codes[:, k] - 7) * sc[:, k // 32].astype(np.float64)
        assert np.array_equal(y[0], want), k
        assert np.array_equal(S[0], np.abs(want))


def test_closed_form_constant_codes(oracle):
    """All codes c and all scales s: y = (c - 7) * s * sum_k x_k."""
    rng = np.random.default_rng(11)
    N, K = 4, 256
    x = synth.activations(rng, 3, K)
    xs = x.astype(np.float64).sum(axis=1)
    for c in range(16):
        wq = np.full((N, K // 8), c * 0x11111111, dtype=np.uint32)
        for s in (0.5, 0.0137, 6.0e-8, 0.0):
            sc = np.full((N, K // 32), s, dtype=np.float16)
            sv = float(sc[0, 0])
            y, S = oracle.gemv(wq, sc, x, N, K)
            want = (c - 7) * sv * xs
            assert np.allclose(y, want[:, None], rtol=0, atol=1e-12 * max(1.0, np.abs(S).max()))
            if c == 7 or sv == 0.0:
                assert np.all(y == 0.0)


def test_brute_force_exact_rationals(oracle):
    """2 x 64 activations against 4 x 64 weights in exact rational arithmetic,
    codes read through the hex-digit route, values through Fraction(float)."""
    rng = np.random.default_rng(5)
    M, N, K = 2, 4, 64
    wq = synth.packed_codes(rng, N, K)
    sc = synth.group_scales(rng, N, K)
    x = synth.activations(rng, M, K)
    y, S = oracle.gemv(wq, sc, x, N, K)
    for n in range(N):
        codes = sum((codes_by_hex(int(w)) for w in wq[n]), [])
        wrow = [(codes[k] - 7) * Fraction(float(sc[n, k // 32])) for k in range(K)]
        for m in range(M):
            exact = sum(Fraction(float(x[m, k])) * wrow[k] for k in range(K))
            sabs = sum(abs(Fraction(float(x[m, k])) * wrow[k]) for k in range(K))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 10 ** 12) * sabs
            assert abs(Fraction(S[m, n]) - sabs) <= Fraction(1, 10 ** 12) * sabs


def test_linearity_power_of_two(oracle):
    rng = np.random.default_rng(9)
    N, K = 16, 128
    wq, sc = synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K)
    x = synth.activations(rng, 2, K)
    y1, _ = oracle.gemv(wq, sc, x, N, K)
    y2, _ = oracle.gemv(wq, sc, (x.astype(np.float32) * 2).astype(np.float16), N, K)
    assert np.array_equal(y2, 2 * y1)


def test_row_subset_matches_full(oracle):
    rng = np.random.default_rng(2)
    N, K = 40, 160
    wq, sc = synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K)
    x = synth.activations(rng, 3, K)
    y, S = oracle.gemv(wq, sc, x, N, K)
    rows = np.array([0, 39, 7, 7, 21])
    ys, Ss = oracle.gemv(wq, sc, x, N, K, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(Ss, S[:, rows])


# --------------------------------------------------------------------------
# SiLU and the gate_up epilogue
# --------------------------------------------------------------------------
def test_silu_values(oracle):
    assert oracle.silu(0.0) == 0.0
    # sigmoid(1) = 1 / (1 + 1/e)
    assert abs(oracle.silu(1.0) - 0.7310585786300049) < 1e-15
    for z in (0.3, 1.7, 5.0, 20.0):
        # silu(z) - silu(-z) = z (sigma(z) + sigma(-z) = 1)
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-12 * max(1.0, z)
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    lib = oracle.lib
    for z in (-3.0, -0.5, 0.0, 0.8, 4.0):
        fd = (oracle.silu(z + 1e-6) - oracle.silu(z - 1e-6)) / 2e-6
        assert abs(lib.zo_silu_deriv(z) - fd) < 1e-8


def test_gate_up_equals_two_gemvs(oracle):
    rng = np.random.default_rng(4)
    I, K, M = 24, 96, 3
    wq, sc = synth.packed_codes(rng, 2 * I, K), synth.group_scales(rng, 2 * I, K)
    x = synth.activations(rng, M, K)
    h, Sh, g, u, Sg, Su = oracle.gate_up_silu(wq, sc, x, 2 * I, K, True, parts=True)
    gy, gS = oracle.gemv(wq[0::2], sc[0::2], x, I, K)
    uy, uS = oracle.gemv(wq[1::2], sc[1::2], x, I, K)
    assert np.array_equal(g, gy) and np.array_equal(u, uy)
    assert np.array_equal(Sg, gS) and np.array_equal(Su, uS)
    want = np.vectorize(oracle.silu)(gy) * uy
    assert np.array_equal(h, want)
    # concatenated layout [gate; up] computes the same thing
    wq_c = np.concatenate([wq[0::2], wq[1::2]])
    sc_c = np.concatenate([sc[0::2], sc[1::2]])
    hc, Shc = oracle.gate_up_silu(wq_c, sc_c, x, 2 * I, K, False)
    assert np.array_equal(hc, h) and np.array_equal(Shc, Sh)


def test_gate_up_bar_is_the_first_order_propagation(oracle):
    """S_h is the first-order sensitivity of h = silu(g) u to moves of g and
    u within their scales S_g and S_u: the worst of the four sign patterns
    reaches it, random moves inside never exceed it (SiLU itself is pinned
    above)."""
    rng = np.random.default_rng(13)
    I, K, M = 16, 64, 2
    wq, sc = synth.packed_codes(rng, 2 * I, K), synth.group_scales(rng, 2 * I, K)
    x = synth.activations(rng, M, K)
    h, Sh, g, u, Sg, Su = oracle.gate_up_silu(wq, sc, x, 2 * I, K, True, parts=True)
    t = 1e-7
    for m in range(M):
        for j in range(I):
            def moved(a, b):
                return oracle.silu(g[m, j] + t * a * Sg[m, j]) * (u[m, j] + t * b * Su[m, j])
            worst = max(abs(moved(a, b) - h[m, j]) for a in (-1, 1) for b in (-1, 1)) / t
            assert abs(worst - Sh[m, j]) <= 1e-5 * Sh[m, j]
            for _ in range(3):
                a, b = rng.random(2) * 2 - 1
                assert abs(moved(a, b) - h[m, j]) / t <= Sh[m, j] * (1 + 1e-5)
    # the affine form carries the same propagation of its own scales
    wa, sa, ba = synth.packed_codes(rng, 2 * I, K), synth.group_scales(rng, 2 * I, K), \
        synth.group_scales(rng, 2 * I, K)
    sa, ba = sa[:, : K // 64], ba[:, : K // 64]
    ha, Sha = oracle.gate_up_silu_affine(wa, sa, ba, x, 2 * I, K)
    ya, Sa = oracle.gemv_affine(wa, sa, ba, x, 2 * I, K)
    for m in range(M):
        for j in range(I):
            ga, ua, sga, sua = ya[m, 2 * j], ya[m, 2 * j + 1], Sa[m, 2 * j], Sa[m, 2 * j + 1]
            worst = max(abs(oracle.silu(ga + t * a * sga) * (ua + t * b * sua) - ha[m, j])
                        for a in (-1, 1) for b in (-1, 1)) / t
            assert abs(worst - Sha[m, j]) <= 1e-5 * Sha[m, j]


def test_gate_up_brute_force(oracle):
    """gate_up on one row pair in exact rationals (SiLU through math.exp)."""
    rng = np.random.default_rng(12)
    K = 64
    wq, sc = synth.packed_codes(rng, 2, K), synth.group_scales(rng, 2, K)
    x = synth.activations(rng, 1, K)
    h, _ = oracle.gate_up_silu(wq, sc, x, 2, K, True)
    vals = []
    for n in range(2):
        codes = sum((codes_by_hex(int(w)) for w in wq[n]), [])
        vals.append(sum(Fraction(float(x[0, k])) * (codes[k] - 7) * Fraction(float(sc[n, k // 32]))
                        for k in range(K)))
    g, u = float(vals[0]), float(vals[1])
    want = g / (1 + math.exp(-g)) * u
    assert abs(h[0, 0] - want) <= 1e-13 * max(1.0, abs(want))


# --------------------------------------------------------------------------
# MoE
# --------------------------------------------------------------------------
def _bank(rng, E, N, K):
    return synth.packed_codes(rng, E * N, K), synth.group_scales(rng, E * N, K)


def test_moe_single_slot_is_plain_gemv(oracle):
    rng = np.random.default_rng(21)
    E, I, K, N = 6, 32, 64, 40
    gq, gs = _bank(rng, E, 2 * I, K)
    dq, ds = _bank(rng, E, N, I)
    T = 3
    x = synth.activations(rng, T, K)
    ids = np.array([[4], [0], [5]], dtype=np.int32)
    h, Sh, bad = oracle.moe_gate_up(gq, gs, E, x, 2 * I, K, ids)
    assert bad == 0
    for t in range(T):
        e = ids[t, 0]
        hr, Shr = oracle.gate_up_silu(gq[e * 2 * I:(e + 1) * 2 * I], gs[e * 2 * I:(e + 1) * 2 * I],
                                      x[t:t + 1], 2 * I, K, True)
        assert np.array_equal(h[t, 0], hr[0]) and np.array_equal(Sh[t, 0], Shr[0])
    hf = h.astype(np.float16)
    r = np.ones((T, 1), dtype=np.float32)
    y, S, bad = oracle.moe_down_combine(dq, ds, E, hf, r, N, I, ids)
    assert bad == 0
    for t in range(T):
        e = ids[t, 0]
        yr, Sr = oracle.gemv(dq[e * N:(e + 1) * N], ds[e * N:(e + 1) * N], hf[t, 0][None], N, I)
        assert np.array_equal(y[t], yr[0]) and np.array_equal(S[t], Sr[0])


def test_moe_combine_weighted_sum_and_slot_permutation(oracle):
    rng = np.random.default_rng(22)
    E, N, K, T, top_k = 10, 24, 64, 4, 3
    dq, ds = _bank(rng, E, N, K)
    h = synth.activations(rng, T * top_k, K).reshape(T, top_k, K)
    ids, r = synth.routing(rng, T, E, top_k)
    y, S, bad = oracle.moe_down_combine(dq, ds, E, h, r, N, K, ids)
    assert bad == 0
    for t in range(T):
        acc = np.zeros(N)
        for j in range(top_k):
            e = ids[t, j]
            z, _ = oracle.gemv(dq[e * N:(e + 1) * N], ds[e * N:(e + 1) * N], h[t, j][None], N, K)
            acc += float(r[t, j]) * z[0]
        assert np.allclose(y[t], acc, rtol=0, atol=1e-13 * S[t].max())
    perm = np.array([2, 0, 1])
    y2, S2, _ = oracle.moe_down_combine(dq, ds, E, h[:, perm], r[:, perm], N, K, ids[:, perm])
    assert np.allclose(y2, y, rtol=0, atol=1e-13 * S.max())


def test_moe_invalid_ids_contribute_nothing(oracle):
    rng = np.random.default_rng(23)
    E, N, K, T = 4, 8, 32, 2
    dq, ds = _bank(rng, E, N, K)
    h = synth.activations(rng, T * 2, K).reshape(T, 2, K)
    ids = np.array([[1, 7], [-1, 2]], dtype=np.int32)
    r = np.full((T, 2), 0.5, dtype=np.float32)
    y, S, bad = oracle.moe_down_combine(dq, ds, E, h, r, N, K, ids)
    assert bad == 2
    ids_ok = np.array([[1, 1], [2, 2]], dtype=np.int32)
    r_ok = np.array([[0.5, 0.0], [0.0, 0.5]], dtype=np.float32)
    y2, _, _ = oracle.moe_down_combine(dq, ds, E, h, r_ok, N, K, ids_ok)
    assert np.array_equal(y, y2)


def test_argmax_hand_cases(oracle):
    """The LM-head argmax on rows whose answer is fixed by the definition:
    the position of the largest value, the lowest one on ties, a NaN above
    every number, -inf below every finite number."""
    nan, inf = float("nan"), float("inf")
    rows = [
        ([1.0, 3.0, 2.0], 1),
        ([-5.0, -1.0, -3.0], 1),
        ([2.0, 7.0, 7.0, 1.0, 7.0], 1),           # ties: lowest index
        ([0.0, -0.0], 0),                         # equal values
        ([-inf, -inf, -1e300], 2),
        ([1.0, nan, 5.0, nan], 1),                # NaN counts as the largest
        ([inf, 4.0, inf], 0),
        ([4.0], 0),
    ]
    for vals, want in rows:
        assert oracle.argmax(np.array([vals]))[0] == want, vals
    # a brute-force check on random integer rows with many ties
    rng = np.random.default_rng(7)
    y = rng.integers(-3, 4, size=(50, 37)).astype(np.float64)
    got = oracle.argmax(y)
    for m in range(50):
        mx = max(y[m])
        assert got[m] == min(n for n in range(37) if y[m, n] == mx)


# --------------------------------------------------------------------------
# the MLX affine format: w = s * q + b, one scale and one bias per 64 weights
# --------------------------------------------------------------------------
def _patterned_affine(N, K, seed=4):
    """codes q[n,k] = (5n + k) mod 16, distinct scales and biases per (n, group of 64)."""
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    codes = (5 * n + k) % 16
    rng = np.random.default_rng(seed)
    sc = (rng.random((N, K // 64)) * 0.9 + 0.05).astype(np.float16)
    bi = (rng.random((N, K // 64)) * 2.0 - 1.0).astype(np.float16)
    return codes, pack_codes(codes), sc, bi


def test_affine_one_hot_columns_exact(oracle):
    """x = e_k returns s[n, k // 64] * q[n,k] + b[n, k // 64] exactly, with
    two groups whose scales and biases differ (k = 63 and 64 fall in
    different groups; a group of 32 would not split there)."""
    N, K = 10, 128
    codes, wq, sc, bi = _patterned_affine(N, K)
    for k in range(K):
        x = np.zeros((1, K), dtype=np.float16)
        x[0, k] = 1.0
        y, Sa = oracle.gemv_affine(wq, sc, bi, x, N, K)
        s_, b_ = sc[:, k // 64].astype(np.float64), bi[:, k // 64].astype(np.float64)
        want = s_ * codes[:, k] + b_
        assert np.array_equal(y[0], want), k
        assert np.array_equal(Sa[0], np.abs(s_) * codes[:, k] + np.abs(b_))


def test_affine_closed_form_constant_codes(oracle):
    """All codes c, scales s and biases b: y = (s c + b) * sum_k x_k; zero
    exactly when s c + b = 0 in exact arithmetic."""
    rng = np.random.default_rng(13)
    N, K = 3, 256
    x = synth.activations(rng, 2, K)
    xs = x.astype(np.float64).sum(axis=1)
    for c in (0, 1, 7, 15):
        wq = np.full((N, K // 8), c * 0x11111111, dtype=np.uint32)
        for s_, b_ in ((0.5, -3.5), (0.0137, 0.25), (2.0, 0.0), (0.25, -0.25 * c)):
            sc = np.full((N, K // 64), s_, dtype=np.float16)
            bi = np.full((N, K // 64), b_, dtype=np.float16)
            wv = float(sc[0, 0]) * c + float(bi[0, 0])
            y, Sa = oracle.gemv_affine(wq, sc, bi, x, N, K)
            assert np.allclose(y, (wv * xs)[:, None], rtol=0, atol=1e-12 * max(1.0, Sa.max()))
            if wv == 0.0:
                assert np.all(y == 0.0)


def test_affine_brute_force_exact_rationals(oracle):
    """2 x 128 activations against 3 x 128 affine weights in exact rational
    arithmetic, codes read through the hex-digit route."""
    rng = np.random.default_rng(17)
    M, N, K = 2, 3, 128
    wq = synth.packed_codes(rng, N, K)
    sc = (rng.random((N, K // 64)) * 0.05).astype(np.float16)
    bi = (rng.standard_normal((N, K // 64)) * 0.1).astype(np.float16)
    x = synth.activations(rng, M, K)
    y, Sa = oracle.gemv_affine(wq, sc, bi, x, N, K)
    for n in range(N):
        codes = sum((codes_by_hex(int(w)) for w in wq[n]), [])
        wrow = [Fraction(float(sc[n, k // 64])) * codes[k] + Fraction(float(bi[n, k // 64])) for k in range(K)]
        wabs = [abs(Fraction(float(sc[n, k // 64]))) * codes[k] + abs(Fraction(float(bi[n, k // 64])))
                for k in range(K)]
        for m in range(M):
            exact = sum(Fraction(float(x[m, k])) * wrow[k] for k in range(K))
            sabs = sum(abs(Fraction(float(x[m, k]))) * wabs[k] for k in range(K))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 10 ** 12) * sabs
            assert abs(Fraction(Sa[m, n]) - sabs) <= Fraction(1, 10 ** 12) * sabs


def test_affine_gate_up_brute_force(oracle):
    """h = silu(g) * u over interleaved affine rows, against a direct fp64
    computation from hex-decoded codes."""
    rng = np.random.default_rng(19)
    M, N2, K = 2, 6, 128
    wq = synth.packed_codes(rng, N2, K)
    sc = (rng.random((N2, K // 64)) * 0.05).astype(np.float16)
    bi = (rng.standard_normal((N2, K // 64)) * 0.1).astype(np.float16)
    x = synth.activations(rng, M, K)
    h, Sh = oracle.gate_up_silu_affine(wq, sc, bi, x, N2, K)
    w = np.array([[float(sc[n, k // 64]) * sum((codes_by_hex(int(v)) for v in wq[n]), [])[k] + float(bi[n, k // 64])
                   for k in range(K)] for n in range(N2)])
    for m in range(M):
        for j in range(N2 // 2):
            g = float(np.dot(x[m].astype(np.float64), w[2 * j]))
            u = float(np.dot(x[m].astype(np.float64), w[2 * j + 1]))
            want = g / (1.0 + math.exp(-g)) * u
            assert abs(h[m, j] - want) <= 1e-12 * (abs(want) + Sh[m, j] + 1e-300)


def _affine_bank(rng, E, N, K):
    wq = synth.packed_codes(rng, E * N, K)
    sc = (rng.random((E * N, K // 64)) * 0.05).astype(np.float16)
    bi = (rng.standard_normal((E * N, K // 64)) * 0.1).astype(np.float16)
    return wq, sc, bi


def test_affine_moe_single_slot_is_plain_gemv(oracle):
    """One slot per token with router weight 1 reduces both affine MoE stages
    to the (pinned) affine GEMV / gate_up of the chosen expert."""
    rng = np.random.default_rng(31)
    E, I, K, N, T = 5, 32, 128, 24, 3
    gq, gs, gb = _affine_bank(rng, E, 2 * I, K)
    dq, ds, db = _affine_bank(rng, E, N, 2 * I)
    x = synth.activations(rng, T, K)
    ids = np.array([[3], [0], [4]], dtype=np.int32)
    h, Sh, bad = oracle.moe_gate_up_affine(gq, gs, gb, E, x, 2 * I, K, ids)
    assert bad == 0
    for t in range(T):
        e = ids[t, 0]
        sl = slice(e * 2 * I, (e + 1) * 2 * I)
        hr, Shr = oracle.gate_up_silu_affine(gq[sl], gs[sl], gb[sl], x[t:t + 1], 2 * I, K)
        assert np.array_equal(h[t, 0], hr[0]) and np.array_equal(Sh[t, 0], Shr[0])
    hf = synth.activations(rng, T, 2 * I).reshape(T, 1, 2 * I)
    y, S, bad = oracle.moe_down_combine_affine(dq, ds, db, E, hf, np.ones((T, 1), np.float32), N, 2 * I, ids)
    assert bad == 0
    for t in range(T):
        e = ids[t, 0]
        sl = slice(e * N, (e + 1) * N)
        yr, Sr = oracle.gemv_affine(dq[sl], ds[sl], db[sl], hf[t, 0][None], N, 2 * I)
        assert np.array_equal(y[t], yr[0]) and np.array_equal(S[t], Sr[0])


def test_affine_moe_combine_weighted_sum_and_invalid_ids(oracle):
    rng = np.random.default_rng(32)
    E, N, K, T, top_k = 7, 16, 128, 3, 3
    dq, ds, db = _affine_bank(rng, E, N, K)
    h = synth.activations(rng, T * top_k, K).reshape(T, top_k, K)
    ids, r = synth.routing(rng, T, E, top_k)
    y, S, bad = oracle.moe_down_combine_affine(dq, ds, db, E, h, r, N, K, ids)
    assert bad == 0
    for t in range(T):
        acc = np.zeros(N)
        for j in range(top_k):
            e = ids[t, j]
            z, _ = oracle.gemv_affine(dq[e * N:(e + 1) * N], ds[e * N:(e + 1) * N], db[e * N:(e + 1) * N],
                                      h[t, j][None], N, K)
            acc += float(r[t, j]) * z[0]
        assert np.allclose(y[t], acc, rtol=0, atol=1e-13 * S[t].max())
    bad_ids = ids.copy()
    bad_ids[0, 1] = E
    bad_ids[2, 0] = -3
    y2, _, bad = oracle.moe_down_combine_affine(dq, ds, db, E, h, r, N, K, bad_ids)
    assert bad == 2
    r2 = r.copy()
    r2[0, 1] = 0.0
    r2[2, 0] = 0.0
    y3, _, _ = oracle.moe_down_combine_affine(dq, ds, db, E, h, r2, N, K, ids)
    assert np.allclose(y2, y3, rtol=0, atol=1e-13 * S.max())


# --------------------------------------------------------------------------
# GEMV + residual add + RMSNorm (the add-norm step at the O / down tails)
# --------------------------------------------------------------------------
def test_add_rmsnorm_zero_weights_closed_form(oracle):
    """All codes 7 (W = 0): r is the residual exactly and out is its RMSNorm,
    computed here with fsum / sqrt from the definition (eps matters)."""
    rng = np.random.default_rng(41)
    M, N, K = 3, 37, 64
    wq = np.full((N, K // 8), 0x77777777, np.uint32)
    sc = synth.group_scales(rng, N, K)
    x = synth.activations(rng, M, K)
    res = synth.activations(rng, M, N)
    gam = (rng.random(N) * 2 - 0.5).astype(np.float16)
    eps = 0.25
    r, out, S, Tn = oracle.gemv_add_rmsnorm(wq, sc, x, res, gam, eps, N, K)
    for m in range(M):
        rv = [float(v) for v in res[m]]
        assert list(r[m]) == rv
        rms = math.sqrt(math.fsum(v * v for v in rv) / N + eps)
        want = [v / rms * float(g) for v, g in zip(rv, gam)]
        assert np.allclose(out[m], want, rtol=1e-14, atol=0)


def test_add_rmsnorm_zero_residual_is_gemv(oracle):
    rng = np.random.default_rng(42)
    M, N, K = 2, 48, 96
    wq, sc = synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K)
    x = synth.activations(rng, M, K)
    r, out, S, _ = oracle.gemv_add_rmsnorm(wq, sc, x, np.zeros((M, N), np.float16), np.ones(N, np.float16),
                                            1e-6, N, K)
    y, Sy = oracle.gemv(wq, sc, x, N, K)
    assert np.array_equal(r, y) and np.array_equal(S, Sy)


def test_add_rmsnorm_scale_invariance(oracle):
    """eps = 0: doubling every scale and the residual doubles r exactly and
    leaves the normalised output unchanged."""
    rng = np.random.default_rng(43)
    M, N, K = 2, 40, 64
    wq, sc = synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K)
    x, res = synth.activations(rng, M, K), synth.activations(rng, M, N)
    gam = (rng.random(N) + 0.5).astype(np.float16)
    r1, o1, _, _ = oracle.gemv_add_rmsnorm(wq, sc, x, res, gam, 0.0, N, K)
    r2, o2, _, _ = oracle.gemv_add_rmsnorm(wq, (sc.astype(np.float32) * 2).astype(np.float16), x,
                                           (res.astype(np.float32) * 2).astype(np.float16), gam, 0.0, N, K)
    assert np.array_equal(r2, 2 * r1)
    assert np.allclose(o2, o1, rtol=1e-14, atol=0)


def test_add_rmsnorm_brute_force(oracle):
    """r in exact rationals from hex-decoded codes; out from fsum / sqrt."""
    rng = np.random.default_rng(44)
    M, N, K = 2, 5, 64
    wq, sc = synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K)
    x, res = synth.activations(rng, M, K), synth.activations(rng, M, N)
    gam = (rng.random(N) + 0.5).astype(np.float16)
    eps = 1e-3
    r, out, S, _ = oracle.gemv_add_rmsnorm(wq, sc, x, res, gam, eps, N, K)
    for m in range(M):
        rex = []
        for n in range(N):
            codes = sum((codes_by_hex(int(w)) for w in wq[n]), [])
            dot = sum(Fraction(float(x[m, k])) * (codes[k] - 7) * Fraction(float(sc[n, k // 32])) for k in range(K))
            rex.append(dot + Fraction(float(res[m, n])))
        for n in range(N):
            assert abs(Fraction(r[m, n]) - rex[n]) <= Fraction(1, 10 ** 12) * (abs(rex[n]) + Fraction(S[m, n]))
        rms = math.sqrt(math.fsum(float(v) ** 2 for v in rex) / N + eps)
        for n in range(N):
            want = float(rex[n]) / rms * float(gam[n])
            assert abs(out[m, n] - want) <= 1e-12 * (abs(want) + 1e-300)


def test_add_rmsnorm_bound_is_the_first_order_propagation(oracle):
    """T_n bounds how far out[n] moves when every r_j moves by at most its
    GEMV bar e_j (to first order), and the worst sign pattern reaches it up to
    the triangle inequality's slack on the r_n term: a dropped or doubled
    term in T_n fails one of the two."""
    rng = np.random.default_rng(45)
    M, N, K = 2, 24, 64
    wq, sc = synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K)
    x, res = synth.activations(rng, M, K), synth.activations(rng, M, N)
    gam = (rng.random(N) * 2 - 0.5).astype(np.float16)
    eps = 0.05
    r, out, S, Tn = oracle.gemv_add_rmsnorm(wq, sc, x, res, gam, eps, N, K)
    g = gam.astype(np.float64)
    t = 1e-6                                           # a small step keeps second-order terms tiny

    def norm(v):
        return v / math.sqrt(math.fsum(v * v) / N + eps) * g

    for m in range(M):
        e = np.ldexp(np.abs(r[m]), -10) + 1e-4 * S[m] + np.ldexp(1.0, -25)
        rms = math.sqrt(math.fsum(r[m] * r[m]) / N + eps)
        assert np.allclose(norm(r[m]), out[m], rtol=1e-13, atol=0)
        for n in range(N):
            # the sign pattern that moves out[n] the most: d out_n / d r_n has
            # the sign of gamma_n, d out_n / d r_j (j != n) that of
            # -gamma_n r_n r_j; T_n exceeds that pattern's move only by the
            # triangle inequality on the r_n term (2 r_n^2 e_n / (N rms^2))
            d = -np.sign(r[m]) * np.sign(r[m, n]) * e
            d[n] = e[n]
            worst = abs(norm(r[m] + t * d)[n] - out[m, n]) / t
            assert worst <= Tn[m, n] * (1 + 1e-6)
            slack = 2 * abs(g[n]) / rms * r[m, n] ** 2 * e[n] / (N * rms * rms)
            assert abs(worst - (Tn[m, n] - slack)) <= 1e-4 * Tn[m, n]
            for _ in range(4):
                dr = (rng.random(N) * 2 - 1) * e
                assert abs(norm(r[m] + t * dr)[n] - out[m, n]) / t <= Tn[m, n] * (1 + 1e-6)


# --------------------------------------------------------------------------
# QKV projection + RoPE over (i, i + D/2) pairs + the token's K / V rows
# --------------------------------------------------------------------------
def _qkv_case(seed, H=3, Hkv=1, D=8, K=64, M=2):
    rng = np.random.default_rng(seed)
    N = (H + 2 * Hkv) * D
    return rng, synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K), synth.activations(rng, M, K)


def test_qkv_rope_position_zero_is_gemv(oracle):
    H, Hkv, D, K = 3, 1, 8, 64
    rng, wq, sc, x = _qkv_case(51, H, Hkv, D, K)
    o = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, 10000.0, [0, 0])
    y, S = oracle.gemv(wq, sc, x, (H + 2 * Hkv) * D, K)
    assert np.array_equal(o["q"], y[:, :H * D])
    assert np.array_equal(o["k"], y[:, H * D:(H + Hkv) * D])
    assert np.array_equal(o["v"], y[:, (H + Hkv) * D:])


def test_qkv_rope_rotation_closed_form(oracle):
    """Each Q / K pair rotated by pos * base^(-2i/D), computed here with
    math.pow / cos / sin from the GEMV outputs (V untouched)."""
    H, Hkv, D, K = 2, 2, 16, 64
    rng, wq, sc, x = _qkv_case(52, H, Hkv, D, K, M=3)
    pos, base = [3, 17, 250], 500.0
    o = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, base, pos)
    y, _ = oracle.gemv(wq, sc, x, (H + 2 * Hkv) * D, K)
    half = D // 2
    for m in range(3):
        for hb in range(H + Hkv):
            for i in range(half):
                a, b = y[m, hb * D + i], y[m, hb * D + i + half]
                th = pos[m] * math.pow(base, -2.0 * i / D)
                want = (a * math.cos(th) - b * math.sin(th), a * math.sin(th) + b * math.cos(th))
                out, h = (o["q"], hb) if hb < H else (o["k"], hb - H)
                got = (out[m, h * D + i], out[m, h * D + i + half])
                assert abs(got[0] - want[0]) <= 1e-12 * (abs(a) + abs(b)) + 1e-300
                assert abs(got[1] - want[1]) <= 1e-12 * (abs(a) + abs(b)) + 1e-300
        assert np.array_equal(o["v"][m], y[m, (H + Hkv) * D:])


def test_qkv_rope_rotations_compose_and_keep_norms(oracle):
    """Rotating at p1 + p2 equals rotating the p1 result by p2's angles, and
    every pair keeps its length."""
    H, Hkv, D, K = 2, 1, 12, 64
    rng, wq, sc, x = _qkv_case(53, H, Hkv, D, K, M=1)
    base, p1, p2 = 10000.0, 7, 30
    o0 = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, base, [0])
    o1 = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, base, [p1])
    o12 = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, base, [p1 + p2])
    half = D // 2
    for name in ("q", "k"):
        for h in range(o1[name].shape[1] // D):
            for i in range(half):
                a0, b0 = o0[name][0, h * D + i], o0[name][0, h * D + i + half]
                a1, b1 = o1[name][0, h * D + i], o1[name][0, h * D + i + half]
                assert abs(math.hypot(a1, b1) - math.hypot(a0, b0)) <= 1e-12 * math.hypot(a0, b0) + 1e-300
                th = p2 * math.pow(base, -2.0 * i / D)
                want = (a1 * math.cos(th) - b1 * math.sin(th), a1 * math.sin(th) + b1 * math.cos(th))
                got = (o12[name][0, h * D + i], o12[name][0, h * D + i + half])
                assert abs(got[0] - want[0]) <= 1e-11 * math.hypot(a0, b0) + 1e-300
                assert abs(got[1] - want[1]) <= 1e-11 * math.hypot(a0, b0) + 1e-300


def _rope_pairs_golden():
    rows = []
    with open(os.path.join(GOLDEN, "rope_pairs.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(tuple(int(v) for v in line.split()))
    return rows


def test_qkv_rope_pairs_golden(oracle):
    """One nonzero projection output at a time (every code 7 but one 8, x
    one-hot): after the rotation at position 1 exactly that dimension and its
    partner from the golden table are nonzero in a Q or K head, and a V head
    keeps the one value where it was."""
    rows = _rope_pairs_golden()
    D = rows[0][0]
    H, Hkv, K = 1, 1, 32
    N = (H + 2 * Hkv) * D
    sc = np.full((N, K // 32), 0.5, np.float16)
    x = np.zeros((1, K), np.float16)
    x[0, 0] = 1.0
    for d, dim, partner in rows:
        assert d == D
        for hb in range(H + 2 * Hkv):
            wq = np.full((N, K // 8), 0x77777777, np.uint32)
            wq[hb * D + dim, 0] = 0x77777778              # element 0: code 8, weight +0.5
            o = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, 10000.0, [1])
            out = o["q"] if hb < H else (o["k"] if hb < H + Hkv else o["v"])
            h = hb if hb < H else (hb - H if hb < H + Hkv else hb - H - Hkv)
            head = out[0, h * D:(h + 1) * D]
            nz = set(np.flatnonzero(head).tolist())
            assert nz == ({dim, partner} if hb < H + Hkv else {dim}), (hb, dim, sorted(nz))
            assert np.count_nonzero(out) == len(nz)       # nothing outside this head
            assert abs(math.hypot(head[dim], head[partner]) - 0.5) <= 1e-15


def test_qkv_rope_frequency_schedule(oracle):
    """The angle of each pair, read back from the output of a single nonzero
    projection value (atan2 of the pair): pair 0 turns by exactly pos
    radians, and each next pair turns base^(2/D) times slower (a geometric
    schedule), at position 1 where no angle wraps."""
    H, Hkv, D, K = 1, 1, 16, 32
    N, half, base = (H + 2 * Hkv) * D, D // 2, 500.0
    sc = np.full((N, 1), 0.5, np.float16)
    x = np.zeros((1, K), np.float16)
    x[0, 0] = 1.0
    for pos in (1, 2):
        angles = []
        for i in range(half):
            wq = np.full((N, K // 8), 0x77777777, np.uint32)
            wq[i, 0] = 0x77777778                          # q row i: value +0.5
            q = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, base, [pos])["q"][0]
            angles.append(math.atan2(q[i + half], q[i]))
        assert abs(angles[0] - pos) <= 1e-15 * pos
        if pos == 1:
            for i in range(half - 1):
                assert abs(angles[i] / angles[i + 1] - base ** (2.0 / D)) <= 1e-12


def test_qkv_rope_bar_covers_the_pair(oracle):
    """The bar of a rotated output, 2^-10 A + 1e-4 S over its pair, covers
    the worst move of the rotation when a and b move within their own GEMV
    bars (|cos| e_a + |sin| e_b); a V output keeps its row's GEMV bar."""
    H, Hkv, D, K = 2, 1, 16, 64
    rng, wq, sc, x = _qkv_case(54, H, Hkv, D, K, M=3)
    pos, base = [0, 5, 900], 10000.0
    o = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, base, pos)
    y, S = oracle.gemv(wq, sc, x, (H + 2 * Hkv) * D, K)
    e = np.ldexp(np.abs(y), -10) + 1e-4 * S
    half = D // 2
    for m in range(3):
        for hb in range(H + Hkv):
            name, h = ("q", hb) if hb < H else ("k", hb - H)
            for i in range(half):
                ra, rb = hb * D + i, hb * D + i + half
                th = pos[m] * math.pow(base, -2.0 * i / D)
                move = abs(math.cos(th)) * e[m, ra] + abs(math.sin(th)) * e[m, rb]
                for c in (h * D + i, h * D + i + half):
                    bar = math.ldexp(o["A_" + name][m, c], -10) + 1e-4 * o["S_" + name][m, c]
                    assert move <= bar * (1 + 1e-12)
                    assert bar <= (e[m, ra] + e[m, rb]) * (1 + 1e-12)
        v0 = (H + Hkv) * D
        bar_v = np.ldexp(o["A_v"][m], -10) + 1e-4 * o["S_v"][m]
        assert np.allclose(bar_v, e[m, v0:], rtol=1e-14, atol=0)


# --------------------------------------------------------------------------
# the pins must be able to fail: mutants planted in the oracle (CPU only)
# --------------------------------------------------------------------------
def _pins_pass(o) -> bool:
    try:
        test_nibble_order_golden(o)
        test_one_hot_columns_exact(o)
        test_brute_force_exact_rationals(o)
        test_closed_form_constant_codes(o)
        test_silu_values(o)
        test_gate_up_brute_force(o)
        test_gate_up_bar_is_the_first_order_propagation(o)
        test_argmax_hand_cases(o)
        test_affine_one_hot_columns_exact(o)
        test_affine_closed_form_constant_codes(o)
        test_affine_brute_force_exact_rationals(o)
        test_add_rmsnorm_zero_weights_closed_form(o)
        test_add_rmsnorm_brute_force(o)
        test_add_rmsnorm_bound_is_the_first_order_propagation(o)
        test_qkv_rope_rotation_closed_form(o)
        test_qkv_rope_pairs_golden(o)
        test_qkv_rope_bar_covers_the_pair(o)
        test_qkv_rope_frequency_schedule(o)
        test_moe_single_slot_is_plain_gemv(o)
        test_moe_combine_weighted_sum_and_slot_permutation(o)
        test_moe_invalid_ids_contribute_nothing(o)
        test_affine_moe_single_slot_is_plain_gemv(o)
        test_affine_moe_combine_weighted_sum_and_invalid_ids(o)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("mutant", list(range(1, 19)))
def test_mutants_are_caught(mutant):
    o = oracle_mod.Oracle(mutant)
    assert o.lib.zo_mutant() == mutant
    assert not _pins_pass(o)


def test_real_oracle_passes_mutant_harness(oracle):
    assert oracle.lib.zo_mutant() == 0
    assert _pins_pass(oracle)
