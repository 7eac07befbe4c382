"""Pins of the oracle's ring bookkeeping and attention."""
import itertools
import math

import numpy as np
import pytest

import synth
from oracle import attention, e4m3, quant, rope
from oracle.ring import OracleRing


# --- ring bookkeeping: brute force with a list of slots ----------------------
@pytest.mark.parametrize("S,writes", [(8, [3, 3, 3, 3]), (5, [5, 1, 4, 2, 5]), (7, [1] * 9 + [7, 6])])
def test_slot_map_brute_force(S, writes):
    H, D = 1, 16
    ring = OracleRing(H, D, S, (D,))
    slots = [None] * S            # token id stored in each slot
    wp, filled, tok = 0, 0, 0
    for n in writes:
        ids = np.arange(tok, tok + n)
        v = np.zeros((n, H, D), np.float32)
        v[:, 0, 0] = 1.0
        v[:, 0, 1] = (ids + 1) / 4096.0           # identifies the token after quantisation
        got = ring.write(np.ones((n, H, D), np.float32), v, np.zeros((n, 1), np.int64))
        for i in range(n):                         # the definition, one token at a time
            slots[wp] = tok + i
            assert got[i] == wp
            wp = (wp + 1) % S
            filled = min(filled + 1, S)
        tok += n
        assert ring.wp == wp and ring.n_valid == filled
        deq = quant.dequantize_rows_f64(ring.v_codes, ring.v_scale)[0]
        for s in range(filled):
            want = (slots[s] + 1) / 4096.0
            assert abs(deq[s, 1] - want) <= want * 2 ** -4


def test_write_size_limits():
    ring = OracleRing(1, 16, 4, (16,))
    with pytest.raises(ValueError):
        ring.write(np.zeros((0, 1, 16), np.float32), np.zeros((0, 1, 16), np.float32), np.zeros((0, 1)))
    with pytest.raises(ValueError):
        ring.write(np.zeros((5, 1, 16), np.float32), np.zeros((5, 1, 16), np.float32), np.zeros((5, 1)))
    ring.write(np.ones((4, 1, 16), np.float32), np.ones((4, 1, 16), np.float32), np.zeros((4, 1)))
    assert ring.wp == 0 and ring.n_valid == 4


def test_no_key_rerotated_twice_in_sustained_workload():
    """Appendix G: the window is shorter than the reset period, so no key is
    requantised twice.  Counted on the sustained workload's slot sequence."""
    S, N, period, steps = synth.SLOTS, synth.NEW_TOKENS, synth.RESET_PERIOD, synth.SUSTAINED_STEPS
    assert S < period * N
    count = np.zeros(S, np.int64)           # rerotations since the slot was written
    wp, filled = 0, 0
    for s in range(steps):
        if s > 0 and s % period == 0:
            count[:filled] += 1
            assert count.max() <= 1
        idx = (wp + np.arange(N)) % S
        count[idx] = 0
        wp = (wp + N) % S
        filled = min(filled + N, S)
    count[:filled] += 1
    assert count.max() <= 1


def test_reset_leaves_values_and_non_temporal_axes_alone():
    g = np.random.default_rng(0)
    H, D, S = 2, 64, 32
    dims = (16, 24, 24)
    ring = OracleRing(H, D, S, dims)
    k = g.standard_normal((S, H, D)).astype(np.float32)
    v = g.standard_normal((S, H, D)).astype(np.float32)
    ring.write(k, v, g.integers(0, 50, (S, 3)))
    vc, vs = ring.v_codes.copy(), ring.v_scale.copy()
    before = quant.dequantize_rows_f64(ring.k_codes, ring.k_scale)
    ring.reset_positions(0)                     # R(0) = identity: one requantisation of the same values
    after = quant.dequantize_rows_f64(ring.k_codes, ring.k_scale)
    assert np.array_equal(before, after)
    ring.reset_positions(5)
    assert np.array_equal(vc, ring.v_codes) and np.array_equal(vs, ring.v_scale)
    after = quant.dequantize_rows_f64(ring.k_codes, ring.k_scale)
    # spatial channels only move by the requantisation to the new scale
    sp = e4m3.spacing(ring.k_codes) * ring.k_scale[..., None]
    assert np.all(np.abs(after[..., 16:] - before[..., 16:]) <= sp[..., 16:])


# --- attention ---------------------------------------------------------------
def _loops(q, k, v):
    Nq, H, D = q.shape
    n = k.shape[1]
    out = np.zeros((Nq, H, D))
    for i, h in itertools.product(range(Nq), range(H)):
        logits = [sum(q[i, h, d] * k[h, j, d] for d in range(D)) / math.sqrt(D) for j in range(n)]
        m = max(logits)
        w = [math.exp(t - m) for t in logits]
        z = sum(w)
        for d in range(D):
            out[i, h, d] = sum(w[j] * v[h, j, d] for j in range(n)) / z
    return out


def test_attention_brute_force():
    g = np.random.default_rng(1)
    q = g.standard_normal((3, 2, 4)) * 2
    k = g.standard_normal((2, 5, 4)) * 2
    v = g.standard_normal((2, 5, 4))
    assert np.allclose(attention.attend_f64(q, k, v), _loops(q, k, v), rtol=1e-13, atol=1e-14)


def test_attention_special_cases():
    g = np.random.default_rng(2)
    q = g.standard_normal((4, 3, 8))
    v = g.standard_normal((3, 6, 8))
    # one valid slot -> O = v exactly
    k1 = g.standard_normal((3, 1, 8))
    assert np.array_equal(attention.attend_f64(q, k1, v[:, :1]), np.broadcast_to(v[:, 0][None], (4, 3, 8)))
    # identical keys -> mean of V
    k = np.repeat(g.standard_normal((3, 1, 8)), 6, axis=1)
    assert np.allclose(attention.attend_f64(q, k, v), np.broadcast_to(v.mean(1)[None], (4, 3, 8)), atol=1e-14)
    # q = 0 -> uniform mean
    k = g.standard_normal((3, 6, 8))
    assert np.allclose(attention.attend_f64(np.zeros((4, 3, 8)), k, v),
                       np.broadcast_to(v.mean(1)[None], (4, 3, 8)), atol=1e-14)
    # a permutation of the slots changes nothing
    perm = g.permutation(6)
    assert np.allclose(attention.attend_f64(q, k, v), attention.attend_f64(q, k[:, perm], v[:, perm]),
                       rtol=1e-13, atol=1e-14)
    with pytest.raises(ValueError):
        attention.attend_f64(q, k[:, :0], v[:, :0])


def test_ring_attend_one_slot_is_the_dequantised_value():
    g = np.random.default_rng(3)
    ring = OracleRing(2, 16, 8, (16,))
    k = g.standard_normal((1, 2, 16)).astype(np.float32)
    v = g.standard_normal((1, 2, 16)).astype(np.float32)
    ring.write(k, v, np.array([[5]]))
    q = g.standard_normal((3, 2, 16)).astype(np.float32)
    out = ring.attend(q, np.array([[5], [6], [7]]))
    want = quant.dequantize_rows_f64(ring.v_codes[:, 0], ring.v_scale[:, 0])
    assert np.array_equal(out, np.broadcast_to(want[None], (3, 2, 16)))


def test_ring_attend_is_plain_attention_over_its_cache():
    g = np.random.default_rng(4)
    H, D, S = 2, 32, 16
    ring = OracleRing(H, D, S, (D,))
    for w in range(3):                               # wraps: 24 tokens into 16 slots
        k = g.standard_normal((8, H, D)).astype(np.float32)
        v = g.standard_normal((8, H, D)).astype(np.float32)
        ring.write(k, v, np.arange(8 * w, 8 * w + 8).reshape(8, 1))
    q = g.standard_normal((5, H, D)).astype(np.float32)
    qp = np.arange(20, 25).reshape(5, 1)
    qc, qs = quant.quantize_rows(rope.rope_f32(q, qp, (D,), 10000.0))
    want = _loops(quant.dequantize_rows_f64(qc, qs),
                  quant.dequantize_rows_f64(ring.k_codes, ring.k_scale),
                  quant.dequantize_rows_f64(ring.v_codes, ring.v_scale))
    assert np.allclose(ring.attend(q, qp), want, rtol=1e-12, atol=1e-13)
    sub = ring.attend(q, qp, heads=[1], rows=[0, 3])
    assert np.allclose(sub, want[[0, 3]][:, [1]], rtol=1e-12, atol=1e-13)
