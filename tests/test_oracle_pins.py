"""Pins for the CPU oracle: each checks the oracle against something other than itself.

Sources of truth used here (none of them is the oracle's own code):
  * numpy's binary16 conversions and float16 arithmetic (library routines);
  * torch's CPU float16 multiply, which rounds the exact fp32 product once (library routine);
  * exact rational arithmetic (``fractions.Fraction``) on tiny inputs;
  * closed forms: one-hot rows, all-ones rows, zero scales, constant weights, linearity;
  * for the activation: the identity silu(g) - silu(-g) = g, its limits, and scipy's logistic;
  * handcrafted packed words whose nibble order is known by construction;
  * for NVFP4 weights: torch's float8_e4m3fn -> float conversion (a library routine) for every
    E4M3 pattern, the literal 16-value E2M1 table of the format definition, exact rationals, and
    closed forms (one-hot rows, zero scales, sign flips, the tensor scale's linearity).

The W4A16 definition (4-bit weights, 16-bit activations) follows "RTX 3090 Tested: Qwen's 381
tok/s Myth Busted" (kongchang.com), section "What Exactly Is This Stack"; the product of one
weight read with several activation rows follows "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s"
(ai.satyajit.si), section "One weight read, shared by every stream". The canonical format
(low nibble first, offset 8, fp16 group scales) is the workload's, not the pages'.

``test_planted_mistake_is_caught`` compiles altered copies of the oracle's C source (a dropped
term, a wrong sign, a wrong index, a transposed operand, a wrong rounding ...) and checks that
at least one pin fails for every one of them.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as inputs

RNG_SEED = 1234


# ------------------------------------------------------------------------------ helpers (numpy)
def np_unpack(qweight: np.ndarray) -> np.ndarray:
    """Independent numpy reading of the canonical words: q[k, n] (uint8)."""
    words = np.asarray(qweight).view(np.uint32)
    K8, N = words.shape
    out = np.empty((K8 * 8, N), np.uint8)
    for j in range(8):
        out[j::8, :] = ((words >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out


def np_dequant(qweight: np.ndarray, scales_bits: np.ndarray, group: int) -> np.ndarray:
    """w = float16((q - 8) * s) with numpy float16 arithmetic (one rounding of an exact product)."""
    q = np_unpack(qweight).astype(np.int16) - 8
    s = np.asarray(scales_bits).view(np.float16)
    s_full = np.repeat(s, group, axis=0)
    with np.errstate(all="ignore"):
        return (q.astype(np.float16) * s_full).astype(np.float64)


def f16_bits(values) -> np.ndarray:
    return np.asarray(values, np.float64).astype(np.float16).view(np.uint16)


def random_case(rng, M, K, N, G, scale_kind="mixed"):
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    flat = q.reshape(-1)
    if flat.size >= 16:
        flat[:16] = rng.permutation(16)  # every nibble value present
    if scale_kind == "workload":
        s = 0.002 * (1.0 + rng.random((K // G, N)))
    else:  # varied exponents, signs and a few subnormal scales
        s = rng.choice([-1.0, 1.0], size=(K // G, N)) * np.exp2(rng.uniform(-12, 3, size=(K // G, N)))
        s.reshape(-1)[::7] = 3.0e-6  # subnormal in binary16
    x = rng.standard_normal((M, K)) * np.exp2(rng.integers(-3, 3, size=(M, K)))
    return f16_bits(x), inputs.pack_nibbles(q), f16_bits(s)


def same_float(a: np.ndarray, b: np.ndarray) -> bool:
    """Bit-level equality of float arrays, NaN == NaN, +0 != -0."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(both_nan | eq))


# ------------------------------------------------------------------------------ pins
def pin_half_decode_all(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    assert same_float(o.half_to_double(bits), ref)


def pin_half_encode(o):
    rng = np.random.default_rng(RNG_SEED)
    fin = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    vals = fin.view(np.float16).astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2.0  # exact ties in double
    rand = rng.choice([-1, 1], 20000) * np.exp2(rng.uniform(-30, 17, 20000))
    special = np.array([65504.0, 65519.99, 65520.0, 65536.0, 1e10, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                        2.0 ** -14 - 2.0 ** -25, 2.0 ** -14 - 2.0 ** -26, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11,
                        0.0, -0.0, np.inf, -np.inf, 1e-300, -1e-300])
    allv = np.concatenate([vals, -vals, mids, -mids, rand, special])
    with np.errstate(over="ignore"):
        ref = allv.astype(np.float16).view(np.uint16)
    got = o.double_to_half(allv)
    assert np.array_equal(got, ref)
    assert o.double_to_half(np.array([np.nan]))[0] & 0x7FFF > 0x7C00


def pin_dequant_exhaustive(o):
    """All 16 nibble values x all 65,536 fp16 scale patterns against torch's fp16 multiply."""
    N = 65536
    words = np.empty((2, N), np.uint32)
    words[0, :] = 0x76543210
    words[1, :] = 0xFEDCBA98
    scales = np.arange(N, dtype=np.uint32).astype(np.uint16).reshape(1, N)
    got = o.dequant(words.view(np.int32), scales, 16)
    qm8 = (torch.arange(16) - 8).to(torch.float16).reshape(16, 1)
    s = torch.from_numpy(scales.view(np.int16)).view(torch.float16)
    ref = (qm8 * s).to(torch.float64).numpy()
    assert same_float(got, ref)


def pin_nibble_order(o):
    w = np.array([[0x76543210, 0xFEDCBA98]], np.uint32).view(np.int32)
    q = o.unpack(w)
    assert q[:, 0].tolist() == list(range(8))
    assert q[:, 1].tolist() == list(range(8, 16))


def pin_pack_roundtrip(o):
    rng = np.random.default_rng(RNG_SEED + 1)
    words = rng.integers(0, 2 ** 32, size=(6, 5), dtype=np.uint64).astype(np.uint32).view(np.int32)
    assert np.array_equal(inputs.pack_nibbles(o.unpack(words)), words)
    q = rng.integers(0, 16, size=(48, 7), dtype=np.uint8)
    assert np.array_equal(o.unpack(inputs.pack_nibbles(q)), q)


def pin_bruteforce_fraction(o):
    rng = np.random.default_rng(RNG_SEED + 2)
    for (M, K, N, G) in [(1, 8, 1, 8), (2, 16, 3, 8), (3, 128, 4, 8), (2, 256, 3, 128), (3, 128, 2, 128)]:
        x, qw, sc = random_case(rng, M, K, N, G)
        y, a = o.gemm(x, qw, sc, G, nthreads=1)
        q = np_unpack(qw).astype(np.int64)
        s = sc.view(np.float16).astype(np.float64)
        w = np.empty((K, N), object)
        for k in range(K):
            for n in range(N):
                prod = float(q[k, n] - 8) * s[k // G, n]  # exact in double
                w[k, n] = Fraction(float(np.float64(prod).astype(np.float16)))
        # Fraction has no signed zero, so compare values (0 == -0) here; signs are pinned elsewhere
        assert np.array_equal(o.dequant(qw, sc, G), np.array(w, dtype=np.float64))
        xf = x.view(np.float16).astype(np.float64)
        for m in range(M):
            for n in range(N):
                terms = [Fraction(float(xf[m, k])) * w[k, n] for k in range(K)]
                exact = sum(terms, Fraction(0))
                exact_abs = sum((abs(t) for t in terms), Fraction(0))
                bound = Fraction(K) * Fraction(2) ** -53 * exact_abs
                assert abs(Fraction(float(y[m, n])) - exact) <= bound
                assert abs(Fraction(float(a[m, n])) - exact_abs) <= bound


def pin_exact_dyadic(o):
    """Small integers x and power-of-two scales: every partial sum is exact, so y is bit-exact."""
    rng = np.random.default_rng(RNG_SEED + 3)
    M, K, N, G = 3, 128, 5, 32
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    xi = rng.integers(-8, 9, size=(M, K))
    s = np.exp2(rng.integers(-6, 2, size=(K // G, N)).astype(np.float64))
    y, a = o.gemm(f16_bits(xi), inputs.pack_nibbles(q), f16_bits(s), G, nthreads=1)
    ref = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            ref[m, n] = sum(int(xi[m, k]) * (int(q[k, n]) - 8) * s[k // G, n] for k in range(K))
    assert np.array_equal(y, ref)


def _workload_matrix(K=256, N=64, G=128, seed=7):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s = 0.002 * (1.0 + rng.random((K // G, N)))
    return inputs.pack_nibbles(q), f16_bits(s)


def pin_one_hot(o):
    K, N, G = 256, 64, 128
    qw, sc = _workload_matrix(K, N, G)
    w = np_dequant(qw, sc, G)
    ks = [0, 7, 8, 127, 128, K - 1]
    x = np.zeros((2 * len(ks), K))
    for i, k in enumerate(ks):
        x[i, k] = 1.0
        x[len(ks) + i, k] = -2.0
    y, _ = o.gemm(f16_bits(x), qw, sc, G, nthreads=1)
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], w[k])
        assert np.array_equal(y[len(ks) + i], -2.0 * w[k])


def pin_all_ones(o):
    K, N, G = 256, 64, 128
    qw, sc = _workload_matrix(K, N, G, seed=8)
    w = np_dequant(qw, sc, G)
    y, a = o.gemm(f16_bits(np.ones((1, K))), qw, sc, G, nthreads=1)
    ref = np.sum(w, axis=0)
    assert np.all(np.abs(y[0] - ref) <= 1e-12 * np.sum(np.abs(w), axis=0))
    assert np.allclose(a[0], np.sum(np.abs(w), axis=0), rtol=1e-12, atol=0)


def pin_zero_scales(o):
    rng = np.random.default_rng(RNG_SEED + 4)
    K, N, G = 256, 32, 128
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s = np.zeros((K // G, N))
    s[0, ::2] = -0.0
    x = f16_bits(rng.standard_normal((3, K)))
    y, a = o.gemm(x, inputs.pack_nibbles(q), f16_bits(s), G, nthreads=1)
    assert np.all(y == 0.0) and np.all(a == 0.0)


def pin_constant_weights(o):
    rng = np.random.default_rng(RNG_SEED + 5)
    K, N, G, M = 256, 32, 128, 3
    x = f16_bits(rng.standard_normal((M, K)))
    xs = x.view(np.float16).astype(np.float64)
    sigma = np.float16(0.0031)
    for c in (0, 3, 8, 9, 15):
        q = np.full((K, N), c, np.uint8)
        s = np.full((K // G, N), float(sigma))
        y, _ = o.gemm(x, inputs.pack_nibbles(q), f16_bits(s), G, nthreads=1)
        wc = float(np.float16(c - 8) * sigma)
        ref = wc * xs.sum(axis=1)
        if c == 8:
            assert np.all(y == 0.0)
        assert np.all(np.abs(y - ref[:, None]) <= 1e-12 * abs(wc) * np.abs(xs).sum(axis=1)[:, None])


def pin_linearity(o):
    rng = np.random.default_rng(RNG_SEED + 6)
    K, N, G = 384, 32, 128
    qw, sc = _workload_matrix(K, N, G, seed=9)
    x1 = rng.standard_normal((2, K))
    x2 = rng.standard_normal((2, K))
    al, be = 1.5, -0.75
    y1, a1 = o.gemm_xf64(x1, qw, sc, G, nthreads=1)
    y2, a2 = o.gemm_xf64(x2, qw, sc, G, nthreads=1)
    y3, _ = o.gemm_xf64(al * x1 + be * x2, qw, sc, G, nthreads=1)
    assert np.all(np.abs(y3 - (al * y1 + be * y2)) <= 1e-12 * (abs(al) * a1 + abs(be) * a2))


def pin_sampled_matches_full(o):
    rng = np.random.default_rng(RNG_SEED + 7)
    M, K, N, G = 5, 256, 96, 128
    x, qw, sc = random_case(rng, M, K, N, G, "workload")
    y, a = o.gemm(x, qw, sc, G, nthreads=2)
    ms = rng.integers(0, M, 40)
    ns = rng.integers(0, N, 40)
    ys, as_ = o.gemm_sampled(x, qw, sc, G, ms, ns, nthreads=2)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


def pin_threads_deterministic(o):
    rng = np.random.default_rng(RNG_SEED + 8)
    x, qw, sc = random_case(rng, 4, 512, 64, 128, "workload")
    y1, a1 = o.gemm(x, qw, sc, 128, nthreads=1)
    y4, a4 = o.gemm(x, qw, sc, 128, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(a1, a4)


def pin_repack_positions(o):
    """Single-nibble matrices land where the layout statement says: 128-column tiles (the last
    one w_t = N - 128t wide), word 16t*K + (b*w_t + c)*4 + w, nibble p = 0,4,1,5,2,6,3,7."""
    K, N, G = 96, 224, 32  # tiles of 128 and 96 columns
    pos_of_j = [0, 4, 1, 5, 2, 6, 3, 7]
    for (k, n) in [(0, 0), (1, 0), (2, 5), (7, 31), (8, 32), (33, 1), (95, 127), (61, 40), (0, 128), (95, 223),
                   (37, 150)]:
        q = np.zeros((K, N), np.uint8)
        q[k, n] = 0xA
        wr, _ = o.repack(inputs.pack_nibbles(q), np.zeros((K // G, N), np.uint16), G)
        t, c = n // 128, n % 128
        wt = min(128, N - 128 * t)
        idx = 16 * t * K + ((k // 32) * wt + c) * 4 + (k % 32) // 8
        assert np.count_nonzero(wr) == 1
        assert wr[idx] == np.uint32(0xA << (4 * pos_of_j[k % 8]))
    sc = np.arange(K // G * N, dtype=np.uint16).reshape(K // G, N)
    _, sr = o.repack(np.zeros((K // 8, N), np.int32), sc, G)
    for (g, n) in [(0, 0), (1, 33), (2, 127), (0, 128), (2, 223)]:
        t, c = n // 128, n % 128
        wt = min(128, N - 128 * t)
        assert sr[128 * t * (K // G) + g * wt + c] == sc[g, n]


def pin_repack_roundtrip(o):
    rng = np.random.default_rng(RNG_SEED + 9)
    K, N, G = 256, 352, 64
    words = rng.integers(0, 2 ** 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    sc = rng.integers(0, 2 ** 16, size=(K // G, N), dtype=np.uint32).astype(np.uint16)
    wr, sr = o.repack(words, sc, G)
    qw2, sc2 = o.unrepack(wr, sr, K, N, G)
    assert np.array_equal(qw2, words) and np.array_equal(sc2, sc)


def _gu_bits(g, u):
    """fp16 bits of [gate | up] for float arrays g, u of the same shape [M, I]."""
    return np.concatenate([np.asarray(g, np.float16), np.asarray(u, np.float16)], axis=1).view(np.uint16)


def pin_silu_identity(o):
    # silu(g) - silu(-g) = g for every g (from silu(g) = g * sigma(g) and sigma(-g) = 1 - sigma(g)),
    # and silu(0) = 0: catches a sign error in the exponent and a gate/up swap
    g = np.linspace(-12.0, 12.0, 401).astype(np.float16).astype(np.float64)
    u = np.ones_like(g)
    a_pos, _ = o.silu_mul(_gu_bits(g[None, :], u[None, :]))
    a_neg, _ = o.silu_mul(_gu_bits(-g[None, :], u[None, :]))
    assert np.allclose(a_pos[0] - a_neg[0], g, rtol=1e-14, atol=1e-300)
    assert a_pos[0][g == 0.0].tolist() == [0.0]


def pin_silu_against_library(o):
    # the logistic from scipy (its own implementation), times g and u, on asymmetric data
    from scipy.special import expit

    rng = np.random.default_rng(RNG_SEED + 10)
    g = rng.normal(0.0, 3.0, size=(5, 64)).astype(np.float16).astype(np.float64)
    u = rng.normal(0.0, 2.0, size=(5, 64)).astype(np.float16).astype(np.float64)
    act, half = o.silu_mul(_gu_bits(g, u))
    ref = g * expit(g) * u
    assert np.allclose(act, ref, rtol=1e-13, atol=1e-300)
    # the fp16 result is numpy's round-to-nearest-even of the double value
    assert np.array_equal(half, act.astype(np.float16).view(np.uint16))


def pin_silu_limits(o):
    # silu(e) / e -> 1/2 as e -> 0; silu(g) -> g for large g; u scales the result exactly
    e = 2.0 ** -20
    act, _ = o.silu_mul(_gu_bits([[e, 20.0]], [[1.0, 1.0]]))
    assert abs(act[0, 0] / e - 0.5) < 1e-6
    assert abs(act[0, 1] - 20.0) < 20.0 * 3e-9
    act2, _ = o.silu_mul(_gu_bits([[1.5, -0.75]], [[2.0, 2.0]]))
    act1, _ = o.silu_mul(_gu_bits([[1.5, -0.75]], [[1.0, 1.0]]))
    assert np.array_equal(act2, 2.0 * act1)


# ------------------------------------------------------------------------------ NVFP4 weights
# The 16 E2M1 values as the NVFP4 / OCP microscaling format definition lists them (sign bit 3,
# then exponent and mantissa): a literal table, not derived from the oracle's decoder.
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def pin_e2m1_table(o):
    got = o.e2m1_to_double(np.arange(16))
    assert np.array_equal(got, np.array(E2M1_VALUES))
    assert np.array_equal(np.signbit(got), np.arange(16) >= 8)


def pin_e4m3_all_patterns(o):
    # every E4M3 pattern against torch's float8_e4m3fn -> float32 conversion (a library routine)
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).float().double().numpy()
    got = o.e4m3_to_double(bits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _nvfp4_case(rng, M, K, N):
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s8 = rng.integers(0, 0x7F, size=(K // 16, N)).astype(np.uint8)  # all finite positive patterns
    x = rng.normal(0.0, 1.0, size=(M, K)).astype(np.float16)
    return q, s8, x


def _frac_e2m1(c):
    return Fraction(E2M1_VALUES[c]) if c not in (0, 8) else Fraction(0)


def _frac_e4m3(b):
    return Fraction(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item())


def pin_nvfp4_bruteforce_fraction(o):
    # y = g * sum_k x * e2m1 * e4m3(s[k // 16]) in exact rationals; the oracle's fp64 sum of exact
    # products over K = 32..64 terms is within a few ulps
    rng = np.random.default_rng(RNG_SEED + 40)
    for (M, K, N, g) in [(1, 32, 2, 0.25), (2, 48, 3, 1.0), (3, 64, 2, 3.0)]:
        q, s8, x = _nvfp4_case(rng, M, K, N)
        qw = inputs.pack_nibbles(q)
        y, a = o.gemm_nvfp4(x.view(np.uint16), qw, s8, g)
        for m in range(M):
            for n in range(N):
                exact = sum(Fraction(float(x[m, k])) * _frac_e2m1(int(q[k, n])) * _frac_e4m3(int(s8[k // 16, n]))
                            for k in range(K))
                exact *= Fraction(g)
                absx = Fraction(g) * sum(abs(Fraction(float(x[m, k])) * _frac_e2m1(int(q[k, n])) *
                                             _frac_e4m3(int(s8[k // 16, n]))) for k in range(K))
                assert abs(Fraction(y[m, n]) - exact) <= Fraction(2) ** -48 * (absx + 1)
                assert abs(Fraction(a[m, n]) - absx) <= Fraction(2) ** -48 * (absx + 1)


def pin_nvfp4_one_hot(o):
    # x = e_k returns g * e2m1(q[k, :]) * e4m3(s[k // 16, :]) exactly, at block edges too
    rng = np.random.default_rng(RNG_SEED + 41)
    K, N, g = 64, 16, 0.5
    q, s8, _ = _nvfp4_case(rng, 1, K, N)
    qw = inputs.pack_nibbles(q)
    ks = [0, 7, 8, 15, 16, 17, 31, 32, 63]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y, _ = o.gemm_nvfp4(x.view(np.uint16), qw, s8, g)
    val = np.array(E2M1_VALUES)
    s_ref = torch.from_numpy(s8.copy()).view(torch.float8_e4m3fn).double().numpy()
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], g * val[q[k]] * s_ref[k // 16])


def pin_nvfp4_zero_scales_sign_and_tensor_scale(o):
    rng = np.random.default_rng(RNG_SEED + 42)
    K, N = 96, 8
    q, s8, x = _nvfp4_case(rng, 3, K, N)
    qw = inputs.pack_nibbles(q)
    xb = x.view(np.uint16)
    y0, _ = o.gemm_nvfp4(xb, qw, np.zeros_like(s8), 1.0)
    assert np.all(y0 == 0.0)
    y1, a1 = o.gemm_nvfp4(xb, qw, s8, 1.0)
    yn, an = o.gemm_nvfp4(xb, inputs.pack_nibbles(q ^ 8), s8, 1.0)  # every sign bit flipped
    assert np.array_equal(yn, -y1) and np.array_equal(an, a1)
    y3, a3 = o.gemm_nvfp4(xb, qw, s8, 3.0)
    assert np.array_equal(y3, 3.0 * y1) and np.array_equal(a3, 3.0 * a1)
    yq, _ = o.gemm_nvfp4(xb, qw, s8, -0.25)
    assert np.array_equal(yq, -0.25 * y1)


def pin_nvfp4_dequant_and_sampled(o):
    rng = np.random.default_rng(RNG_SEED + 43)
    K, N = 128, 24
    q, s8, x = _nvfp4_case(rng, 4, K, N)
    qw = inputs.pack_nibbles(q)
    w = o.dequant_nvfp4(qw, s8)
    s_ref = torch.from_numpy(s8.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(w, np.array(E2M1_VALUES)[q] * np.repeat(s_ref, 16, axis=0))
    # every weight is exactly an fp16 number (the product of 2 and 4 significant bits)
    assert np.array_equal(w.astype(np.float16).astype(np.float64), w)
    y, a = o.gemm_nvfp4(x.view(np.uint16), qw, s8, 0.125)
    ms = np.array([0, 3, 1, 2, 3]); ns = np.array([0, 23, 5, 11, 17])
    ys, as_ = o.gemm_nvfp4_sampled(x.view(np.uint16), qw, s8, 0.125, ms, ns)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


def pin_nvfp4_repack(o):
    # natural nibble order inside the words of the int4 device layout, scales as equal-valued fp16
    K, N = 64, 160
    q = np.zeros((K, N), np.uint8)
    s8 = np.zeros((K // 16, N), np.uint8)
    for (k, n, v) in [(0, 0, 1), (1, 0, 2), (7, 0, 3), (8, 0, 4), (33, 5, 5), (63, 127, 6), (9, 130, 7)]:
        q[k, n] = v
    s8[1, 3] = 0x38
    s8[3, 150] = 0x01
    wr, sr = o.repack_nvfp4(inputs.pack_nibbles(q), s8)
    # tile 0 (128 wide): word ((b * 128 + c) * 4 + w), nibble k % 8
    assert wr[0] == (1 | 2 << 4 | 3 << 28) and wr[1] == 4
    assert wr[(1 * 128 + 5) * 4 + 0] == 5 << 4
    assert wr[(1 * 128 + 127) * 4 + 3] == 6 << 28
    # tile 1 (32 wide) starts at word 16 * 1 * K
    assert wr[16 * K + (0 * 32 + 2) * 4 + 1] == 7 << 4
    # scales: tile 0 [K/16][128], tile 1 [K/16][32] after 128 * K/16 entries
    assert sr[1 * 128 + 3] == np.float16(1.0).view(np.uint16)
    assert sr[128 * (K // 16) + 3 * 32 + 22] == np.float16(2.0 ** -9).view(np.uint16)
    qw2, s82 = o.unrepack_nvfp4(wr, sr, K, N)
    assert np.array_equal(qw2, inputs.pack_nibbles(q)) and np.array_equal(s82, s8)
    rng = np.random.default_rng(RNG_SEED + 44)
    q, s8, _ = _nvfp4_case(rng, 1, 256, 96)
    qw = inputs.pack_nibbles(q)
    wr, sr = o.repack_nvfp4(qw, s8)
    qw2, s82 = o.unrepack_nvfp4(wr, sr, 256, 96)
    assert np.array_equal(qw2, qw) and np.array_equal(s82, s8)


# ------------------------------------------------------------------------------ W4A8 (int8 activations)
def _quantize_numpy(x16):
    """The per-token decision restated in numpy binary32 (an implementation independent of the C one)."""
    xf = x16.astype(np.float32)
    amax = np.max(np.abs(xf), axis=1).astype(np.float32)
    sx = (amax / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (xf / sx[:, None]).astype(np.float32)
    xq = np.where(amax[:, None] > 0, np.clip(np.rint(r), -127, 127), 0).astype(np.int8)
    return xq, sx


def pin_w4a8_quantize(o):
    K = 16
    rows = np.zeros((5, K), np.float32)
    rows[0, :7] = [127, -127, 5, -6, 0, 64, -1]            # amax 127: sx = 1, xq = x
    rows[1, :9] = [127, 2.5, 3.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5]  # ties go to even
    # rows[2] stays zero: sx = 0, xq = 0
    rows[3, :4] = [1016, -8, 24, -1000]                     # amax 127 * 8: sx = 8, xq = x / 8
    rows[4, :3] = [-100, 50, 20]                            # the largest magnitude is negative
    x16 = rows.astype(np.float16)
    xq, sx = o.quantize_x_int8(x16.view(np.uint16))
    assert sx[0] == 1.0 and np.array_equal(xq[0], rows[0].astype(np.int8))
    assert np.array_equal(xq[1, :9], [127, 2, 4, -2, 0, 0, 2, -2, 126])
    assert sx[2] == 0.0 and not xq[2].any()
    assert sx[3] == 8.0 and np.array_equal(xq[3, :4], [127, -1, 3, -125])
    assert sx[4] == np.float32(100) / np.float32(127) and xq[4, 0] == -127
    rng = np.random.default_rng(RNG_SEED + 50)
    for scale in (1.0, 1e-3, 300.0):
        x = (rng.standard_normal((6, 320)) * scale).astype(np.float16)
        x[1] = (rng.standard_cauchy(320) * scale).clip(-60000, 60000).astype(np.float16)  # heavy tails
        xq, sx = o.quantize_x_int8(x.view(np.uint16))
        xq_ref, sx_ref = _quantize_numpy(x)
        assert np.array_equal(sx, sx_ref) and np.array_equal(xq, xq_ref)


def _w4a8_case(rng, M, K, N, G):
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    # fp16 scales of both signs and several binades (a signed scale checks |s| in the tolerance sum)
    sc = (rng.uniform(0.5, 1.0, size=(K // G, N)) * rng.choice([-1.0, 1.0], size=(K // G, N)) *
          2.0 ** rng.integers(-12, 2, size=(K // G, N))).astype(np.float16)
    xq = rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    sx = rng.uniform(1e-3, 0.1, size=M).astype(np.float32)
    return q, sc, xq, sx


def pin_w4a8_bruteforce_fraction(o):
    # y = sx * sum_g s_g * sum_{k in g} (q - 8) xq in exact rationals
    rng = np.random.default_rng(RNG_SEED + 51)
    for (M, K, N, G) in [(1, 16, 3, 8), (2, 32, 2, 16), (3, 48, 2, 8)]:
        q, sc, xq, sx = _w4a8_case(rng, M, K, N, G)
        qw = inputs.pack_nibbles(q)
        y, a = o.gemm_w4a8(xq, sx, qw, sc.view(np.uint16), G)
        for m in range(M):
            for n in range(N):
                terms = [Fraction(float(sx[m])) * Fraction(float(sc[k // G, n])) * (int(q[k, n]) - 8) * int(xq[m, k])
                         for k in range(K)]
                exact, absx = sum(terms), sum(abs(t) for t in terms)
                assert abs(Fraction(y[m, n]) - exact) <= Fraction(2) ** -48 * (absx + 1)
                assert abs(Fraction(a[m, n]) - absx) <= Fraction(2) ** -48 * (absx + 1)


def pin_w4a8_matches_w4a16_when_exact(o):
    # power-of-two scales make (q - 8) * s exact in fp16, and x = j / 8 with max |j| = 127 gives
    # sx = 1/8 exactly and xq = j: then W4A8 and the (separately pinned) W4A16 oracle compute the same
    # sum of exact dyadic products and must agree to the last bit
    rng = np.random.default_rng(RNG_SEED + 52)
    M, K, N, G = 3, 256, 24, 64
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    sc = (2.0 ** rng.integers(-10, -2, size=(K // G, N)) * rng.choice([-1.0, 1.0], size=(K // G, N))).astype(np.float16)
    j = rng.integers(-126, 127, size=(M, K))
    j[:, 5] = 127
    x = (j / 8.0).astype(np.float16)
    qw = inputs.pack_nibbles(q)
    xq, sx = o.quantize_x_int8(x.view(np.uint16))
    assert np.all(sx == 0.125) and np.array_equal(xq, j.astype(np.int8))
    y8, a8 = o.gemm_w4a8(xq, sx, qw, sc.view(np.uint16), G)
    y16, a16 = o.gemm(x.view(np.uint16), qw, sc.view(np.uint16), G)
    assert np.array_equal(y8, y16) and np.array_equal(a8, a16)


def pin_w4a8_one_hot(o):
    # x = e_k: xq = 127 e_k, sx = fl32(1/127), y = sx * s[k/G] * 127 (q[k] - 8)
    rng = np.random.default_rng(RNG_SEED + 53)
    K, N, G = 64, 12, 16
    q, sc, _, _ = _w4a8_case(rng, 1, K, N, G)
    qw = inputs.pack_nibbles(q)
    ks = [0, 15, 16, 17, 47, 63]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    xq, sx = o.quantize_x_int8(x.view(np.uint16))
    assert np.all(sx == np.float32(1) / np.float32(127))
    y, _ = o.gemm_w4a8(xq, sx, qw, sc.view(np.uint16), G)
    for i, k in enumerate(ks):
        assert xq[i, k] == 127 and np.count_nonzero(xq[i]) == 1
        for n in range(N):
            exact = Fraction(float(sx[i])) * Fraction(float(sc[k // G, n])) * 127 * (int(q[k, n]) - 8)
            assert abs(Fraction(y[i, n]) - exact) <= Fraction(2) ** -51 * abs(exact)


def pin_w4a8_zero_sign_linearity_sampled(o):
    rng = np.random.default_rng(RNG_SEED + 54)
    M, K, N, G = 4, 128, 20, 32
    q, sc, xq, sx = _w4a8_case(rng, M, K, N, G)
    qw = inputs.pack_nibbles(q)
    s16 = sc.view(np.uint16)
    y0, _ = o.gemm_w4a8(xq, sx, qw, np.zeros_like(s16), G)
    assert np.all(y0 == 0.0)
    y, a = o.gemm_w4a8(xq, sx, qw, s16, G)
    yn, an = o.gemm_w4a8((-xq.astype(np.int16)).astype(np.int8), sx, qw, s16, G)
    assert np.array_equal(yn, -y) and np.array_equal(an, a)
    y2, a2 = o.gemm_w4a8(xq, (2 * sx).astype(np.float32), qw, s16, G)
    assert np.array_equal(y2, 2 * y) and np.array_equal(a2, 2 * a)
    ms = np.array([0, 3, 1, 2, 3]); ns = np.array([0, 19, 5, 11, 7])
    ys, as_ = o.gemm_w4a8_sampled(xq, sx, qw, s16, G, ms, ns)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


PINS = [pin_half_decode_all, pin_half_encode, pin_dequant_exhaustive, pin_nibble_order, pin_pack_roundtrip,
        pin_bruteforce_fraction, pin_exact_dyadic, pin_one_hot, pin_all_ones, pin_zero_scales,
        pin_constant_weights, pin_linearity, pin_sampled_matches_full, pin_threads_deterministic,
        pin_repack_positions, pin_repack_roundtrip, pin_silu_identity, pin_silu_against_library, pin_silu_limits,
        pin_e2m1_table, pin_e4m3_all_patterns, pin_nvfp4_bruteforce_fraction, pin_nvfp4_one_hot,
        pin_nvfp4_zero_scales_sign_and_tensor_scale, pin_nvfp4_dequant_and_sampled, pin_nvfp4_repack,
        pin_w4a8_quantize, pin_w4a8_bruteforce_fraction, pin_w4a8_matches_w4a16_when_exact, pin_w4a8_one_hot,
        pin_w4a8_zero_sign_linearity_sampled]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_mod):
    pin(oracle_mod.load())


# ------------------------------------------------------------------------------ planted mistakes
MUTANTS = {
    "dropped_term": ("for (int k = 0; k < K; ++k) {\n        double p = xrow[k] * col[k];",
                     "for (int k = 1; k < K; ++k) {\n        double p = xrow[k] * col[k];"),
    "wrong_sign": ("double prod = (double)(q - 8) * s;", "double prod = (double)(8 - q) * s;"),
    "wrong_zero_point": ("double prod = (double)(q - 8) * s;", "double prod = (double)(q - 7) * s;"),
    "wrong_group_index": ("scales[(size_t)(k / G) * (size_t)N", "scales[(size_t)(k / (2 * G)) * (size_t)N"),
    "nibble_high_first": ("(word >> (4 * (k % 8)))", "(word >> (28 - 4 * (k % 8)))"),
    "ties_away_from_zero": ("r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "r = fl + 1.0;"),
    "unrounded_weight": ("return w4o_half_to_double(w4o_double_to_half(prod));", "return prod;"),
    "subnormal_flush_decode": ("v = ldexp((double)m, -24);", "v = 0.0;"),
    "subnormal_encode": ("if (ex < -14) ex = -14;", ""),
    "transposed_output": ("&y[(size_t)m * N + n], &absy[(size_t)m * N + n]",
                          "&y[(size_t)n * M + m], &absy[(size_t)n * M + m]"),
    "shifted_x_row": ("column_dot(x + (size_t)m * K,", "column_dot(x + (size_t)m,"),
    "abs_not_abs": ("aacc += fabs(p);", "aacc += p;"),
    "layout_positions": ("kPosOfJ[8] = {0, 4, 1, 5, 2, 6, 3, 7};", "kPosOfJ[8] = {0, 1, 2, 3, 4, 5, 6, 7};"),
    "layout_transposed_tile": ("((size_t)b * wt + c) * 4 + w;", "((size_t)c * (K / 32) + b) * 4 + w;"),
    "silu_exponent_sign": ("g / (1.0 + exp(-g)) * u;", "g / (1.0 + exp(g)) * u;"),
    "silu_gate_up_swapped": ("gu[(size_t)m * 2 * I + i]);\n            const double u = w4o_half_to_double(gu[(size_t)m * 2 * I + I + i]);",
                             "gu[(size_t)m * 2 * I + I + i]);\n            const double u = w4o_half_to_double(gu[(size_t)m * 2 * I + i]);"),
    "silu_without_up": ("g / (1.0 + exp(-g)) * u;", "g / (1.0 + exp(-g));"),
    "silu_sigmoid_only": ("g / (1.0 + exp(-g)) * u;", "1.0 / (1.0 + exp(-g)) * u;"),
    "e2m1_subnormal_as_normal": ("double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                                 "double v = ldexp(1.0 + 0.5 * m, e - 1);"),
    "e4m3_wrong_bias": ("else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    "nvfp4_block_of_32": ("scales8[(size_t)(k / 16) * (size_t)N + (size_t)n]);",
                          "scales8[(size_t)(k / 32) * (size_t)N + (size_t)n]);"),
    "nvfp4_tensor_scale_dropped": ("y[(size_t)m * N + n] = g * s;", "y[(size_t)m * N + n] = s;"),
    "nvfp4_repack_permuted": ("wr[weight_word_index(K, N, k, n)] |= q << (4 * (k % 8));",
                              "wr[weight_word_index(K, N, k, n)] |= q << (4 * kPosOfJ[k % 8]);"),
    "w4a8_offset_7": ("(int64_t)(qcol[k] - 8)", "(int64_t)(qcol[k] - 7)"),
    "w4a8_ties_away_from_zero": ("float t = nearbyintf(r);", "float t = roundf(r);"),
    "w4a8_scale_over_128": ("float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    "w4a8_amax_signed": ("float v = fabsf((float)w4o_half_to_double(row[k]));",
                         "float v = (float)w4o_half_to_double(row[k]);"),
    "w4a8_group_index": ("scales[(size_t)g * (size_t)N + (size_t)n]", "scales[(size_t)(g / 2) * (size_t)N + (size_t)n]"),
    "w4a8_sx_dropped": ("*y = sxm * acc;", "*y = acc;"),
    "w4a8_signed_scale_in_abs": ("aacc += fabs(s) * (double)iabs;", "aacc += s * (double)iabs;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, oracle_mod):
    old, new = MUTANTS[name]
    src = oracle_mod.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    bad = oracle_mod.load_from_source(src.replace(old, new), str(tmp_path))
    caught = []
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"


def test_tolerance_helper_flags_errors(oracle_mod):
    y_ref = np.array([1.0, -2.0, 0.0, 3.0])
    a_ref = np.array([2.0, 2.0, 1.0, 4.0])
    bound = 2.0 ** -10 * (np.abs(y_ref) + a_ref)
    ok, worst, nbad = oracle_mod.within_tolerance(y_ref + 0.99 * bound, y_ref, a_ref)
    assert ok and worst < 1.0 and nbad == 0
    ok, worst, nbad = oracle_mod.within_tolerance(y_ref + 1.01 * bound, y_ref, a_ref)
    assert not ok and nbad == 4
    ok, _, nbad = oracle_mod.within_tolerance(np.array([np.nan, -2.0, 0.0, 3.0]), y_ref, a_ref)
    assert not ok and nbad == 1
