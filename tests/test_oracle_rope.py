"""Pins of the oracle's RoPE, its fp32 version and the delta rotation."""
import math
import os

import numpy as np
import pytest

from oracle import attention, quant, rope, e4m3
from oracle.ring import OracleRing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_hand.txt")


def test_frequencies_closed_form():
    w = rope.frequencies(8, 10000.0)
    assert np.allclose(w, [1.0, 0.1, 0.01, 0.001], rtol=1e-15, atol=0)
    w = rope.frequencies(4, 100.0)
    assert np.allclose(w, [1.0, 0.1], rtol=1e-15, atol=0)


def test_hand_worked_vectors():
    """tests/golden/rope_hand.txt: cases worked by hand from the rotation
    formula (x0 cos t - x1 sin t, x0 sin t + x1 cos t)."""
    n = 0
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split("|")
        dims = tuple(int(t) for t in f[0].split())
        base = float(f[1])
        pos = np.array([[int(t) for t in f[2].split()]])
        x = np.array([[[float(t) for t in f[3].split()]]])
        want = np.array([eval(t, {"cos": math.cos, "sin": math.sin}) for t in f[4].split()])
        got = rope.rope_f64(x, pos, dims, base)[0, 0]
        assert np.allclose(got, want, rtol=0, atol=1e-15), line
        got32 = rope.rope_f32(x.astype(np.float32), pos, dims, base)[0, 0]
        assert np.allclose(got32, want, rtol=0, atol=4e-7 * np.abs(x).sum()), line
        n += 1
    assert n >= 5


def test_norm_preserved_per_pair():
    g = np.random.default_rng(0)
    x = g.standard_normal((64, 3, 128))
    pos = g.integers(-40000, 40000, (64, 3))
    dims = (32, 48, 48)
    y = rope.rope_f64(x, pos, dims, 10000.0)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(ny, nx, rtol=1e-12, atol=0)


@pytest.mark.parametrize("dims", [(64,), (16, 24, 24)])
def test_dot_product_depends_on_relative_position_only(dims):
    g = np.random.default_rng(1)
    q = g.standard_normal((1, 1, 64))
    k = g.standard_normal((1, 1, 64))
    p = g.integers(-500, 500, (1, len(dims)))
    pk = g.integers(-500, 500, (1, len(dims)))
    ref = np.sum(rope.rope_f64(q, p, dims, 10000.0) * rope.rope_f64(k, pk, dims, 10000.0))
    for _ in range(5):
        s = g.integers(-3000, 3000, (1, len(dims)))
        got = np.sum(rope.rope_f64(q, p + s, dims, 10000.0) * rope.rope_f64(k, pk + s, dims, 10000.0))
        assert abs(got - ref) <= 1e-11 * (1 + abs(ref))
    # and it does change with the relative position
    s = np.zeros((1, len(dims)), np.int64)
    s[0, 0] = 1
    other = np.sum(rope.rope_f64(q, p + s, dims, 10000.0) * rope.rope_f64(k, pk, dims, 10000.0))
    assert abs(other - ref) > 1e-3


def test_fp32_rope_within_rounding_bound_of_fp64():
    g = np.random.default_rng(2)
    x = g.standard_normal((200, 4, 128)).astype(np.float32) * 8
    pos = g.integers(-32768, 32768, (200, 1))
    y32 = rope.rope_f32(x, pos, (128,), 10000.0).astype(np.float64)
    y64 = rope.rope_f64(x.astype(np.float64), pos, (128,), 10000.0)
    pair = np.repeat(np.abs(x[..., 0::2]) + np.abs(x[..., 1::2]), 2, axis=-1).astype(np.float64)
    # cos/sin rounded (2 x 2^-24), two products (2^-24 each), one sum (2^-24)
    assert np.all(np.abs(y32 - y64) <= 4 * 2.0 ** -24 * pair + 1e-30)


def test_numpy_cos_agrees_with_libm():
    g = np.random.default_rng(3)
    t = g.integers(-40000, 40000, 20000) * rope.frequencies(128, 10000.0)[g.integers(0, 64, 20000)]
    assert np.array_equal(np.cos(t), [math.cos(v) for v in t])
    assert np.array_equal(np.sin(t), [math.sin(v) for v in t])


def test_table_rows_match_direct_angles():
    tab = rope.rope_table_f32(64, 10000.0, -5, 20)
    c, s = rope.cos_sin_f32(np.arange(-5, 15), rope.frequencies(64, 10000.0))
    assert np.array_equal(tab[..., 0], c) and np.array_equal(tab[..., 1], s)
    assert tab[5, 0, 0] == 1.0 and tab[5, 0, 1] == 0.0           # position 0


@pytest.mark.parametrize("dims", [(128,), (32, 48, 48)])
def test_delta_rotation_equals_fresh_rope_f64(dims):
    g = np.random.default_rng(4)
    k = g.standard_normal((50, 2, 128))
    p = g.integers(0, 32000, (50, len(dims)))
    d = 42 * 757
    rot = rope.rotate_temporal_f64(rope.rope_f64(k, p, dims, 10000.0), d, dims[0], 10000.0)
    shifted = p.copy()
    shifted[:, 0] -= d
    fresh = rope.rope_f64(k, shifted, dims, 10000.0)
    # the two sides form angles (p - d) w and p w - d w: each rounded in fp64,
    # so they differ by a few ulps of the largest angle (|p| + |d| radians)
    ang = (np.abs(p).max() + d) * 2.0 ** -52 * 4
    assert np.allclose(rot, fresh, rtol=0, atol=ang * np.abs(k).max() * 2)
    assert np.allclose(rot[..., dims[0]:], rope.rope_f64(k, p, dims, 10000.0)[..., dims[0]:], rtol=0, atol=0)
    # the fp32 delta table is the fp64 rotation rounded once
    c, s = rope.delta_cos_sin_f32(d, dims[0], 10000.0)
    th = -d * rope.frequencies(dims[0], 10000.0)
    assert np.array_equal(c, np.cos(th).astype(np.float32))
    assert np.array_equal(s, np.sin(th).astype(np.float32))


def test_fp8_rerotated_key_close_to_fresh_quantisation():
    """In FP8 the rotation identity holds up to the roundings: the rerotated
    dequantised key differs from the exact key at p-d by at most the first
    rounding (rotated) plus the second rounding plus fp32 arithmetic."""
    g = np.random.default_rng(5)
    H, D, S = 4, 128, 256
    ring = OracleRing(H, D, S, (D,))
    k = g.standard_normal((S, H, D)).astype(np.float32)
    v = g.standard_normal((S, H, D)).astype(np.float32)
    pos = np.arange(1000, 1000 + S).reshape(S, 1)
    ring.write(k, v, pos)
    scale1 = ring.k_scale.copy()
    codes1 = ring.k_codes.copy()
    d = 777
    ring.reset_positions(d)
    got = quant.dequantize_rows_f64(ring.k_codes, ring.k_scale)              # [H,S,D]
    exact = np.transpose(rope.rope_f64(k.astype(np.float64), pos - d, (D,), 10000.0), (1, 0, 2))
    # first rounding: half a spacing per element, rotation mixes the pair
    sp1 = e4m3.spacing(codes1) * scale1[..., None]
    e1 = np.repeat(np.sqrt(sp1[..., 0::2] ** 2 + sp1[..., 1::2] ** 2), 2, -1) / 2
    sp2 = e4m3.spacing(ring.k_codes) * ring.k_scale[..., None] / 2
    bound = e1 + sp2 + 1e-5 * np.abs(exact) + 1e-6
    assert np.all(np.abs(got - exact) <= bound)
    # against a fresh quantisation at p-d (its own scale grid) the gap is at
    # most those roundings plus the fresh one
    fresh = OracleRing(H, D, S, (D,))
    fresh.write(k, v, pos - d)
    fr = quant.dequantize_rows_f64(fresh.k_codes, fresh.k_scale)
    sp3 = e4m3.spacing(fresh.k_codes) * fresh.k_scale[..., None] / 2
    assert np.all(np.abs(got - fr) <= bound + sp3)


def test_invalid_combination_ring_with_read_time_rope_in_slot_order():
    """Runway Characters paper §4.1: re-applying RoPE in physical slot order is
    only right while slot == position; once the ring wraps it permutes the
    keys' temporal positions.  Pinned here on the fp64 definition."""
    g = np.random.default_rng(6)
    S, N, D = 8, 4, 8
    k_raw = g.standard_normal((16, 1, D))
    v = g.standard_normal((16, 1, D))
    q = g.standard_normal((1, 1, D))

    def attend_write_time(n_tok):
        pos = np.arange(n_tok).reshape(-1, 1)
        keep = np.arange(max(0, n_tok - S), n_tok)
        kk = rope.rope_f64(k_raw[keep], pos[keep], (D,), 100.0)
        qq = rope.rope_f64(q, np.array([[n_tok]]), (D,), 100.0)
        return attention.attend_f64(qq, np.transpose(kk, (1, 0, 2)), np.transpose(v[keep], (1, 0, 2)))

    def attend_read_time_slot_order(n_tok):
        keep = np.arange(max(0, n_tok - S), n_tok)
        slots = keep % S                       # where each token sits in the ring
        kk = rope.rope_f64(k_raw[keep], slots.reshape(-1, 1), (D,), 100.0)
        qq = rope.rope_f64(q, np.array([[n_tok]]), (D,), 100.0)
        return attention.attend_f64(qq, np.transpose(kk, (1, 0, 2)), np.transpose(v[keep], (1, 0, 2)))

    assert np.allclose(attend_write_time(8), attend_read_time_slot_order(8), atol=1e-12)
    assert not np.allclose(attend_write_time(12), attend_read_time_slot_order(12), atol=1e-3)
