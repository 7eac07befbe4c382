"""Pins of the oracle's per-head scales fixed once per session.

Runway Characters paper, §4.3 "FP8 at write" and Appendix G: K and V are
quantised with per-(cache, head) scales, set once per session from the
absolute maximum of what the first steps wrote, times a margin of 1.5; values
beyond the range saturate; a position reset dequantises the window keys with
their head's scale, rotates them in fp32, clamps them to the FP8 range and
requantises them with the same scale.
"""
import numpy as np
import pytest
import torch

from oracle import attention, e4m3, quant, rope
from oracle.ring import OracleRing


def _calibrated_ring(g, H=3, D=32, S=24, n=16, dims=None, margin=1.5):
    dims = dims or (D,)
    ring = OracleRing(H, D, S, dims, scale_mode="static")
    k = g.standard_normal((n, H, D)).astype(np.float32)
    v = (g.standard_normal((n, H, D)) * np.array([0.5, 2.0, 8.0])[None, :H, None]).astype(np.float32)
    pos = np.arange(n).reshape(n, 1) if len(dims) == 1 else g.integers(0, 20, (n, len(dims)))
    ring.write(k[:9], v[:9], pos[:9])
    ring.write(k[9:], v[9:], pos[9:])
    kr = rope.rope_f32(k, pos, dims, 10000.0)
    return ring, kr, v


def test_static_scale_is_a_plain_cast_when_margin_times_amax_is_448():
    """margin * amax = 448 gives scale 1 and inv 1: the codes are the plain
    e4m3 cast of the values (PyTorch's float8_e4m3fn, inside the range)."""
    scale, inv = quant.static_scale(np.float32(256.0), margin=1.75)
    assert scale == np.float32(1.0) and inv == np.float32(1.0)
    g = np.random.default_rng(20)
    x = (g.standard_normal((64, 32)) * 60).astype(np.float32)
    x = np.clip(x, -440, 440)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = quant.quantize_rows_fixed(x, np.full(64, inv, np.float32))
    assert np.array_equal(got, want)


def test_static_scale_properties():
    amax = np.array([0.0, 1e-30, 0.37, 3.0, 1234.5], np.float32)
    scale, inv = quant.static_scale(amax, margin=1.5)
    assert scale[0] == 0 and inv[0] == 0
    a = 1.5 * amax[1:].astype(np.float64)
    # scale * 448 is 1.5 * amax and inv * 1.5 * amax is 448, each within two fp32 roundings
    assert np.all(np.abs(scale[1:].astype(np.float64) * 448 / a - 1) <= 2 * 2.0 ** -24)
    assert np.all(np.abs(inv[1:].astype(np.float64) * a / 448 - 1) <= 2 * 2.0 ** -24)


def test_values_beyond_the_range_saturate_and_inv_zero_gives_plus_zero():
    x = np.array([[1.0, -1.0, 3.0, -3.0, 0.5, -0.0, 2.9, 0.0]], np.float32)
    codes = quant.quantize_rows_fixed(x, np.array([np.float32(448.0 / 2.0)]))
    vals = e4m3.decode(codes)[0]
    assert vals[2] == 448.0 and vals[3] == -448.0 and vals[6] == 448.0   # 3 * 224, 2.9 * 224 > 448
    assert vals[0] == 224.0 and vals[1] == -224.0 and vals[4] == 112.0
    z = quant.quantize_rows_fixed(x, np.array([np.float32(0.0)]))
    assert np.all(z == 0)


def test_calibration_sets_one_scale_per_head_from_the_written_maxima():
    g = np.random.default_rng(21)
    ring, kr, v = _calibrated_ring(g)
    assert np.array_equal(ring.cal_amax_k, np.abs(kr).max(axis=(0, 2)))
    assert np.array_equal(ring.cal_amax_v, np.abs(v).max(axis=(0, 2)))
    old_k = quant.dequantize_rows_f64(ring.k_codes[:, :16], ring.k_scale[:, :16])
    old_v = quant.dequantize_rows_f64(ring.v_codes[:, :16], ring.v_scale[:, :16])
    ring.calibrate(1.5)
    ks, _ = quant.static_scale(ring.cal_amax_k, 1.5)
    vs, _ = quant.static_scale(ring.cal_amax_v, 1.5)
    # every valid slot now carries its head's scale, bit for bit
    assert np.array_equal(ring.k_scale[:, :16].view(np.uint32), np.repeat(ks[:, None], 16, 1).view(np.uint32))
    assert np.array_equal(ring.v_scale[:, :16].view(np.uint32), np.repeat(vs[:, None], 16, 1).view(np.uint32))
    # the margin leaves headroom: the largest value maps to 448 / 1.5 -> no code above 288
    for codes in (ring.k_codes[:, :16], ring.v_codes[:, :16]):
        assert np.abs(e4m3.decode(codes)).max() <= 288.0
    # each value moved by at most half a spacing of its new code (plus fp32 rounding)
    for codes, scales, old in ((ring.k_codes, ring.k_scale, old_k), (ring.v_codes, ring.v_scale, old_v)):
        new = quant.dequantize_rows_f64(codes[:, :16], scales[:, :16])
        sp = e4m3.spacing(codes[:, :16]) * scales[:, :16, None].astype(np.float64)
        assert np.all(np.abs(new - old) <= sp / 2 + 1e-6 * np.abs(old) + 1e-30)


def test_writes_after_calibration_use_the_fixed_scales_and_saturate():
    g = np.random.default_rng(22)
    H, D = 3, 32
    ring, kr, v = _calibrated_ring(g, H=H, D=D)
    ring.calibrate(1.5)
    ks, _ = quant.static_scale(ring.cal_amax_k, 1.5)
    vs, _ = quant.static_scale(ring.cal_amax_v, 1.5)
    k_new = np.zeros((2, H, D), np.float32)
    v_new = np.zeros((2, H, D), np.float32)
    v_new[0, :, 0] = 3.0 * ring.cal_amax_v            # beyond 1.5 x the calibration maximum
    v_new[0, :, 1] = -3.0 * ring.cal_amax_v
    v_new[0, :, 2] = 0.25 * ring.cal_amax_v
    slots = ring.write(k_new, v_new, np.array([[16], [17]]))
    s0 = slots[0]
    vals = e4m3.decode(ring.v_codes[:, s0])
    assert np.all(vals[:, 0] == 448.0) and np.all(vals[:, 1] == -448.0)
    dq = vals[:, 2] * vs.astype(np.float64)
    sp = e4m3.spacing(ring.v_codes[:, s0, 2]) * vs.astype(np.float64)
    assert np.all(np.abs(dq - 0.25 * ring.cal_amax_v.astype(np.float64)) <= sp / 2 + 1e-6)
    assert np.array_equal(ring.k_scale[:, s0].view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(ring.v_scale[:, s0].view(np.uint32), vs.view(np.uint32))
    assert np.all(e4m3.decode(ring.k_codes[:, s0]) == 0)             # zero K row: +-0 (sign kept)


def test_reset_keeps_the_scales_and_clamps():
    g = np.random.default_rng(23)
    H, D = 2, 16
    ring = OracleRing(H, D, 8, (D,), scale_mode="static")
    k = g.standard_normal((4, H, D)).astype(np.float32)
    ring.write(k, k, np.zeros((4, 1), np.int64))
    ring.calibrate(1.5)
    amax = ring.cal_amax_k
    # a key whose first temporal pair is (1.4 a, 1.4 a): turned by 1 radian it
    # has a component 1.4 a (sin 1 + cos 1) = 1.93 a, beyond the 1.5 a the
    # scale holds
    big = np.zeros((1, H, D), np.float32)
    big[0, :, 0] = 1.4 * amax
    big[0, :, 1] = 1.4 * amax
    big[0, :, 2:] = g.standard_normal((H, D - 2)).astype(np.float32) * 0.3
    slot = int(ring.write(big, big, np.zeros((1, 1), np.int64))[0])
    sk_before = ring.k_scale.copy()
    codes_before = ring.k_codes.copy()
    d = -1                      # omega_0 = 1: R(-d) turns temporal pair 0 by +1 radian
    ring.reset_positions(d)
    assert np.array_equal(sk_before.view(np.uint32), ring.k_scale.view(np.uint32))
    # pair 0 of the planted key: x0 cos1 - x1 sin1 and x0 sin1 + x1 cos1 with x0 = x1:
    # the second is 1.4 a (sin 1 + cos 1) = 1.93 a > 1.5 a -> saturated
    vals = e4m3.decode(ring.k_codes[:, slot])
    assert np.all(vals[:, 1] == 448.0)
    # every other value is the rotated dequantised key within half a spacing
    c, s = rope.delta_cos_sin_f32(d, D, 10000.0)
    x = quant.dequantize_rows(codes_before[:, :5], sk_before[:, :5])
    want = rope.rotate_temporal_f32(x, c, s, D).astype(np.float64)
    got = quant.dequantize_rows_f64(ring.k_codes[:, :5], ring.k_scale[:, :5])
    sp = e4m3.spacing(ring.k_codes[:, :5]) * ring.k_scale[:, :5, None].astype(np.float64)
    lim = 448.0 * np.broadcast_to(ring.k_scale[:, :5, None], got.shape).astype(np.float64)
    clamped = np.abs(want) > lim
    ok = np.abs(got - want) <= sp / 2 + 1e-6 * np.abs(want)
    assert np.all(ok | clamped)
    assert np.all(np.abs(got[clamped]) == lim[clamped])
    assert clamped.sum() >= H


def test_static_ring_attention_is_plain_attention_over_its_cache():
    g = np.random.default_rng(24)
    ring, _, _ = _calibrated_ring(g, H=2, D=32, S=24, n=16)
    ring.calibrate(1.5)
    k = g.standard_normal((12, 2, 32)).astype(np.float32)             # wraps: 28 tokens into 24 slots
    ring.write(k, k * 0.5, np.arange(16, 28).reshape(12, 1))
    q = g.standard_normal((3, 2, 32)).astype(np.float32)
    qp = np.arange(25, 28).reshape(3, 1)
    qc, qs = quant.quantize_rows(rope.rope_f32(q, qp, (32,), 10000.0))
    want = attention.attend_f64(quant.dequantize_rows_f64(qc, qs),
                                quant.dequantize_rows_f64(ring.k_codes, ring.k_scale),
                                quant.dequantize_rows_f64(ring.v_codes, ring.v_scale))
    assert np.allclose(ring.attend(q, qp), want, rtol=1e-12, atol=1e-13)


def test_static_mode_call_rules():
    z = np.ones((2, 1, 16), np.float32)
    p = np.zeros((2, 1), np.int64)
    with pytest.raises(ValueError):
        OracleRing(1, 16, 8, (16,), scale_mode="rolling")
    token = OracleRing(1, 16, 8, (16,))
    token.write(z, z, p)
    with pytest.raises(ValueError):
        token.calibrate()                           # token scales: nothing to calibrate
    ring = OracleRing(1, 16, 8, (16,), scale_mode="static")
    with pytest.raises(ValueError):
        ring.calibrate()                            # nothing written yet
    ring.write(z, z, p)
    with pytest.raises(ValueError):
        ring.reset_positions(3)                     # calibrate before the first reset
    ring.calibrate()
    with pytest.raises(ValueError):
        ring.calibrate()                            # once per session
    ring.reset_positions(3)


def test_static_workloads_replay_on_the_oracle():
    """The seeded static-scale workloads follow the call rules; the x3 step
    drives some values past the calibrated range (saturated codes appear)."""
    import synth
    wl = synth.static_scales_tiny()
    sh = wl.shape
    ring = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base, n_global=sh.n_global,
                      scale_mode=sh.scale_mode)
    kinds = []
    for op in wl.ops:
        kinds.append(type(op).__name__)
        if isinstance(op, synth.WriteGlobal):
            ring.write_global(synth.to_f32(op.k), synth.to_f32(op.v), op.pos)
        elif isinstance(op, synth.Write):
            ring.write(synth.to_f32(op.k), synth.to_f32(op.v), op.pos)
        elif isinstance(op, synth.Calibrate):
            ring.calibrate(op.margin)
        elif isinstance(op, synth.Reset):
            ring.reset_positions(op.d)
        else:
            assert np.all(np.isfinite(ring.attend(synth.to_f32(op.q), op.pos)))
    assert kinds.count("Calibrate") == 1 and kinds.count("Reset") == 1
    assert kinds.index("Calibrate") < kinds.index("Reset")
    vals = np.abs(e4m3.decode(np.concatenate([ring.k_codes, ring.v_codes])))
    assert (vals == 448.0).any()
