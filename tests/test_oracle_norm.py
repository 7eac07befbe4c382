"""Pins of the oracle's RMS normalisation (oracle/norm.py).

Runway Characters paper, §4.4 "Fused pre-attention" and Appendix G: Q and K
are RMS-normalised (squares in fp32) before RoPE and the FP8 write.
"""
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import norm


def test_rn32_matches_numpy_on_doubles_and_rounds_ties_to_even():
    g = np.random.default_rng(30)
    x = g.standard_normal(2000) * np.exp2(g.uniform(-100, 100, 2000))
    for v in x:
        assert norm.rn32(Fraction(float(v))) == np.float32(v)
    # exact midpoints between adjacent fp32 values: ties to the even significand
    one = Fraction(1)
    assert norm.rn32(one + Fraction(1, 2 ** 24)) == np.float32(1.0)                  # 1 is even
    assert norm.rn32(one + Fraction(3, 2 ** 24)) == np.float32(1.0 + 2.0 ** -22)     # not 1 + 2^-23 (odd)
    # a hair off a midpoint decides the direction
    assert norm.rn32(one + Fraction(1, 2 ** 24) + Fraction(1, 2 ** 90)) == np.float32(1.0 + 2.0 ** -23)
    assert norm.rn32(-(one + Fraction(1, 2 ** 24) - Fraction(1, 2 ** 90))) == np.float32(-1.0)


def test_sum_of_squares_is_exact_then_rounded_once():
    # small integers: the exact sum is an integer
    g = np.random.default_rng(31)
    row = g.integers(-3, 4, 128).astype(np.float32)
    assert norm.sum_sq_f32(row) == np.float32(np.sum(row.astype(np.int64) ** 2))
    # the order of the terms cannot change it
    x = (g.standard_normal(128) * np.exp2(g.uniform(-8, 8, 128))).astype(np.float32)
    assert norm.sum_sq_f32(x).view(np.uint32) == norm.sum_sq_f32(x[::-1]).view(np.uint32)
    assert norm.sum_sq_f32(x).view(np.uint32) == norm.sum_sq_f32(g.permutation(x)).view(np.uint32)
    # (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24 is an fp32 midpoint; + 2^-80 puts the
    # exact sum above it, which fp64 (then fp32, ties to even) would round down
    a, b = np.float32(1 + 2.0 ** -12), np.float32(2.0 ** -40)
    assert float(a) ** 2 == 1 + 2.0 ** -11 + 2.0 ** -24
    assert np.float32(math.fsum([float(a) ** 2, float(b) ** 2])) == np.float32(1 + 2.0 ** -11)
    assert norm.sum_sq_f32(np.array([a, b])) == np.float32(1 + 2.0 ** -11 + 2.0 ** -23)


def test_rsqrt_is_correctly_rounded():
    for k in range(-60, 61):                             # 1/sqrt(4^k) = 2^-k exactly
        assert norm.rsqrt_rn32(np.float32(4.0 ** k)) == np.float32(2.0 ** -k)
    getcontext().prec = 60
    g = np.random.default_rng(32)
    vs = (g.uniform(0.5, 2.0, 400) * np.exp2(g.integers(-100, 100, 400))).astype(np.float32)
    for v in vs:
        want = norm.rn32(Fraction(Decimal(1) / Decimal(float(v)).sqrt()))      # 60-digit, then one rounding
        assert norm.rsqrt_rn32(v) == want
        # from a start one or two ulps off, the exact tests still land on it
        for start in (np.nextafter(want, np.float32(0)), np.nextafter(want, np.float32(np.inf)),
                      np.nextafter(np.nextafter(want, np.float32(0)), np.float32(0))):
            assert norm.rsqrt_rn32(v, start=start) == want
    with pytest.raises(ValueError):
        norm.rsqrt_rn32(np.float32(0.0))


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(33)
    x = (g.standard_normal(5000) * np.exp2(g.uniform(-60, 60, 5000))).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]      # ties
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(norm.round_bf16(x).view(np.uint32), want.view(np.uint32))


def _bf16(g, shape, scale=1.0):
    return norm.round_bf16((g.standard_normal(shape) * scale).astype(np.float32))


def test_rms_norm_closed_forms_and_symmetries():
    g = np.random.default_rng(34)
    H, D = 3, 64
    # a constant row c (a power of two) with gamma = 1: +-1 exactly
    for c in (2.0 ** -20, 0.5, 8.0, 2.0 ** 30):
        row = np.full((1, D), c, np.float32)
        assert np.all(norm.rms_norm_bf16(row, 1.0, eps=1e-30 * c * c) == 1.0)
        assert np.all(norm.rms_norm_bf16(-row, 1.0, eps=1e-30 * c * c) == -1.0)
    x = _bf16(g, (5, H, D), 3.0)
    gamma = _bf16(g, (H, D)) + np.float32(1.0)
    y = norm.rms_norm_bf16(x, gamma, eps=0.0)
    # scale invariance by powers of two (with eps = 0)
    for k in (-7, 3, 20):
        assert np.array_equal(norm.rms_norm_bf16(x * np.float32(2.0 ** k), gamma, eps=0.0).view(np.uint32),
                              y.view(np.uint32))
    # odd symmetry, and gamma doubled doubles the output
    assert np.array_equal(norm.rms_norm_bf16(-x, gamma, eps=0.0), -y)
    assert np.array_equal(norm.rms_norm_bf16(x, 2 * gamma, eps=0.0), 2 * y)
    # permuting the channels (and gamma with them) permutes the output
    perm = g.permutation(D)
    assert np.array_equal(norm.rms_norm_bf16(x[..., perm], gamma[:, perm], eps=0.0), y[..., perm])
    # a zero row stays zero (eps > 0)
    assert np.all(norm.rms_norm_bf16(np.zeros((2, D), np.float32), 1.0, eps=1e-6) == 0)


@pytest.mark.parametrize("D", [64, 128])
def test_rms_norm_against_the_formula_in_fp64(D):
    g = np.random.default_rng(35)
    H = 4
    x = _bf16(g, (16, H, D), 2.0)
    x[0, 0] *= np.float32(1e-3)                     # rows where eps matters
    gamma = _bf16(g, (H, D)) * np.float32(0.5) + np.float32(1.0)
    for eps in (1e-6, 1.0):
        y = norm.rms_norm_bf16(x, gamma, eps=eps).astype(np.float64)
        xd = x.astype(np.float64)
        exact = xd / np.sqrt((xd ** 2).mean(-1, keepdims=True) + np.float32(eps)) * gamma.astype(np.float64)
        # one bf16 rounding (half of 2^-7 relative) plus a few fp32 roundings
        assert np.all(np.abs(y - exact) <= np.abs(exact) * (2.0 ** -8 + 2.0 ** -20) + 1e-30)


def test_ring_norm_option_is_the_norm_then_the_plain_call():
    """write / write_global / attend with norm = (gamma, eps) act on
    rms_norm_bf16 of K (or Q); V is left as it is."""
    from oracle.ring import OracleRing
    g = np.random.default_rng(36)
    H, D, G, W = 2, 32, 3, 8
    gk, gq = _bf16(g, (H, D)) + np.float32(1.0), _bf16(g, (H, D)) + np.float32(1.0)
    a = OracleRing(H, D, G + W, (D,), n_global=G)
    b = OracleRing(H, D, G + W, (D,), n_global=G)
    kg, vg = _bf16(g, (G, H, D), 4.0), _bf16(g, (G, H, D))
    k, v = _bf16(g, (6, H, D), 4.0), _bf16(g, (6, H, D))
    a.write_global(kg, vg, np.arange(-G, 0).reshape(G, 1), norm_k=(gk, 1e-6))
    b.write_global(norm.rms_norm_bf16(kg, gk, 1e-6), vg, np.arange(-G, 0).reshape(G, 1))
    a.write(k, v, np.arange(6).reshape(6, 1), norm_k=(gk, 1e-6))
    b.write(norm.rms_norm_bf16(k, gk, 1e-6), v, np.arange(6).reshape(6, 1))
    for name in ("k_codes", "v_codes", "k_scale", "v_scale"):
        assert np.array_equal(getattr(a, name), getattr(b, name))
    q = _bf16(g, (4, H, D), 4.0)
    qp = np.arange(2, 6).reshape(4, 1)
    assert np.array_equal(a.attend(q, qp, norm_q=(gq, 1e-6)), b.attend(norm.rms_norm_bf16(q, gq, 1e-6), qp))
