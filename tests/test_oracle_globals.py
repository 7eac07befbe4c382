"""Pins of the oracle's global slots and window ring.

Runway Characters paper, Introduction ("The model") and Appendix G: each cache
holds 1,246 global slots written once per session and a ring of six latent
frames of 757 tokens (5,788 slots in all); attention reads every slot; a
position reset rotates the window keys only, since the global tokens'
positions do not depend on the window.
"""
import numpy as np
import pytest

from oracle import attention, e4m3, quant, rope
from oracle.ring import OracleRing


def _tagged(ids, H, D):
    """K of ones, V whose channel 1 identifies the token after quantisation."""
    n = len(ids)
    v = np.zeros((n, H, D), np.float32)
    v[:, :, 0] = 1.0
    v[:, :, 1] = (np.asarray(ids)[:, None] + 1) / 4096.0
    return np.ones((n, H, D), np.float32), v


def _token_in_slot(ring, s):
    deq = quant.dequantize_rows_f64(ring.v_codes, ring.v_scale)[0]
    return deq[s, 1] * 4096.0 - 1.0


@pytest.mark.parametrize("S,G,writes", [(12, 5, [3, 3, 3, 3, 1]), (9, 1, [8, 1, 8, 2]), (20, 13, [7, 1, 6, 5])])
def test_global_and_window_slot_map_brute_force(S, G, writes):
    """A list of slots filled one token at a time against the ring's slots."""
    H, D = 1, 16
    W = S - G
    ring = OracleRing(H, D, S, (D,), n_global=G)
    k, v = _tagged(range(G), H, D)
    assert list(ring.write_global(k, v, np.zeros((G, 1), np.int64))) == list(range(G))
    assert ring.n_valid == G and ring.wp == 0
    model = list(range(G)) + [None] * W          # token id per slot
    wp, tok = 0, G
    for n in writes:
        k, v = _tagged(range(tok, tok + n), H, D)
        got = ring.write(k, v, np.zeros((n, 1), np.int64))
        for i in range(n):
            assert got[i] == G + wp
            model[G + wp] = tok + i
            wp = (wp + 1) % W
        tok += n
        filled = sum(t is not None for t in model)
        assert ring.wp == wp and ring.n_valid == filled
        for s in range(filled):                    # filled slots are 0 .. n_valid-1
            want = model[s]
            assert abs(_token_in_slot(ring, s) - want) <= (want + 1) * 2 ** -4
        assert all(model[s] < G for s in range(G))  # globals never overwritten


def test_frames_fill_whole_slots_at_the_papers_layout():
    """1,246 globals + six 757-token frames: frame f lands in slots
    1246 + (f mod 6) * 757 .. + 756 and the seventh frame replaces the first."""
    G, N, F = 1246, 757, 6
    S = G + F * N
    assert S == 5788
    ring = OracleRing(1, 16, S, (16,), n_global=G)
    z = np.zeros((G, 1, 16), np.float32)
    ring.write_global(z, z, np.zeros((G, 1), np.int64))
    zn = np.zeros((N, 1, 16), np.float32)
    for f in range(2 * F + 1):
        slots = ring.write(zn, zn, np.zeros((N, 1), np.int64))
        start = G + (f % F) * N
        assert np.array_equal(slots, np.arange(start, start + N))
        assert ring.n_valid == min(G + (f + 1) * N, S)
        assert ring.wp == ((f + 1) % F) * N


def test_window_keys_requantised_at_most_once_between_resets_at_the_papers_layout():
    """Appendix G: the window (6 latents) is shorter than the reset period
    (42 steps), so no window key is rotated twice; globals are never rotated.
    Counted on the slot sequence of 126 steps with resets every 42."""
    G, N, F, period = 1246, 757, 6, 42
    S = G + F * N
    count = np.zeros(S, np.int64)
    wp, filled = 0, G
    for s in range(126):
        if s > 0 and s % period == 0:
            count[G:filled] += 1
            assert count[G:].max() <= 1 and count[:G].max() == 0
        idx = G + (wp + np.arange(N)) % (S - G)
        count[idx] = 0
        wp = (wp + N) % (S - G)
        filled = min(filled + N, S)


def test_reset_rotates_window_keys_only():
    g = np.random.default_rng(11)
    H, D, G, W = 2, 64, 5, 12
    dims = (32, 16, 16)
    ring = OracleRing(H, D, G + W, dims, n_global=G)
    kg = g.standard_normal((G, H, D)).astype(np.float32)
    vg = g.standard_normal((G, H, D)).astype(np.float32)
    pg = g.integers(-40, 40, (G, 3))
    ring.write_global(kg, vg, pg)
    kw = g.standard_normal((W + 4, H, D)).astype(np.float32)     # wraps: 16 tokens into 12 slots
    vw = g.standard_normal((W + 4, H, D)).astype(np.float32)
    pw = np.stack([100 + np.arange(W + 4), np.arange(W + 4) % 4, np.arange(W + 4) // 4], 1)
    ring.write(kw[:9], vw[:9], pw[:9])
    ring.write(kw[9:], vw[9:], pw[9:])
    gk, gs = ring.k_codes[:, :G].copy(), ring.k_scale[:, :G].copy()
    wk, ws = ring.k_codes[:, G:].copy(), ring.k_scale[:, G:].copy()
    vc, vs = ring.v_codes.copy(), ring.v_scale.copy()
    d = 37
    ring.reset_positions(d)
    # globals and every value: bit for bit unchanged
    assert np.array_equal(gk, ring.k_codes[:, :G]) and np.array_equal(gs.view(np.uint32),
                                                                         ring.k_scale[:, :G].view(np.uint32))
    assert np.array_equal(vc, ring.v_codes) and np.array_equal(vs, ring.v_scale)
    # window slot G + s holds the last token written there; it is now the key
    # at temporal position p - d, within the roundings of a fresh quantisation
    last = {}
    for t in range(W + 4):
        last[t % W] = t
    toks = np.array([last[s] for s in range(W)])
    p_new = pw[toks].copy()
    p_new[:, 0] -= d
    exact = np.transpose(rope.rope_f64(kw[toks].astype(np.float64), p_new, dims, 10000.0), (1, 0, 2))
    got = quant.dequantize_rows_f64(ring.k_codes[:, G:], ring.k_scale[:, G:])
    # the write's rounding (half a spacing of the old code, mixed within each
    # temporal pair by the rotation; spatial pairs are not rotated, but the
    # pair bound covers them) plus the reset's rounding (half a new spacing)
    sp1 = e4m3.spacing(wk) * ws[..., None]
    e1 = np.repeat(np.sqrt(sp1[..., 0::2] ** 2 + sp1[..., 1::2] ** 2), 2, -1) / 2
    sp2 = e4m3.spacing(ring.k_codes[:, G:]) * ring.k_scale[:, G:, None] / 2
    assert np.all(np.abs(got - exact) <= e1 + sp2 + 1e-5 * np.abs(exact) + 1e-6)
    assert not np.array_equal(ring.k_codes[:, G:], np.zeros_like(ring.k_codes[:, G:]))


def test_attention_reads_the_globals_and_the_last_window_tokens():
    """The ring's attention equals plain attention over the G global tokens and
    the last W window tokens, each quantised on its own (slot order aside)."""
    g = np.random.default_rng(12)
    H, D, G, W = 2, 32, 3, 8
    ring = OracleRing(H, D, G + W, (D,), n_global=G)
    ks = g.standard_normal((G + 19, H, D)).astype(np.float32)
    vs = g.standard_normal((G + 19, H, D)).astype(np.float32)
    pos = np.concatenate([np.arange(-G, 0), np.arange(19)]).reshape(-1, 1)
    ring.write_global(ks[:G], vs[:G], pos[:G])
    for a, b in ((G, G + 6), (G + 6, G + 13), (G + 13, G + 19)):
        ring.write(ks[a:b], vs[a:b], pos[a:b])
    keep = np.concatenate([np.arange(G), np.arange(G + 19 - W, G + 19)])
    kc, kq = quant.quantize_rows(rope.rope_f32(ks[keep], pos[keep], (D,), 10000.0))
    vc, vq = quant.quantize_rows(vs[keep])
    kd = np.transpose(quant.dequantize_rows_f64(kc, kq), (1, 0, 2))
    vd = np.transpose(quant.dequantize_rows_f64(vc, vq), (1, 0, 2))
    q = g.standard_normal((4, H, D)).astype(np.float32)
    qp = np.arange(15, 19).reshape(4, 1)
    qc, qs = quant.quantize_rows(rope.rope_f32(q, qp, (D,), 10000.0))
    want = attention.attend_f64(quant.dequantize_rows_f64(qc, qs), kd, vd)
    assert np.allclose(ring.attend(q, qp), want, rtol=1e-12, atol=1e-13)


def test_call_sequence_rules():
    H, D = 1, 16
    z = lambda n: np.zeros((n, H, D), np.float32)  # noqa: E731
    p = lambda n: np.zeros((n, 1), np.int64)       # noqa: E731
    with pytest.raises(ValueError):
        OracleRing(H, D, 8, (D,), n_global=8)      # no window slot left
    ring = OracleRing(H, D, 8, (D,), n_global=3)
    with pytest.raises(ValueError):
        ring.write(z(2), z(2), p(2))               # window before globals
    with pytest.raises(ValueError):
        ring.write_global(z(2), z(2), p(2))        # not exactly n_global tokens
    ring.write_global(z(3), z(3), p(3))
    with pytest.raises(ValueError):
        ring.write_global(z(3), z(3), p(3))        # once per session
    with pytest.raises(ValueError):
        ring.write(z(6), z(6), p(6))               # more than the 5 window slots
    ring.write(z(5), z(5), p(5))
    assert (ring.wp, ring.n_valid) == (0, 8)
    plain = OracleRing(H, D, 8, (D,))
    with pytest.raises(ValueError):
        plain.write_global(z(1), z(1), p(1))       # no global slots


def test_windowed_workloads_are_valid_call_sequences():
    """The seeded global-slot workloads follow the call rules, and every
    position they pass lies inside their RoPE tables."""
    import synth
    wl = synth.windowed_tiny()
    sh = wl.shape
    ring = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base, n_global=sh.n_global)
    n_attend = 0
    for op in wl.ops:
        if isinstance(op, synth.WriteGlobal):
            ring.write_global(synth.to_f32(op.k), synth.to_f32(op.v), op.pos)
        elif isinstance(op, synth.Write):
            ring.write(synth.to_f32(op.k), synth.to_f32(op.v), op.pos)
        elif isinstance(op, synth.Reset):
            ring.reset_positions(op.d)
        else:
            assert np.all(np.isfinite(ring.attend(synth.to_f32(op.q), op.pos)))
            n_attend += 1
        if hasattr(op, "pos"):
            lo, cnt = np.array(sh.pos_min), np.array(sh.pos_count)
            assert np.all(op.pos >= lo) and np.all(op.pos < lo + cnt)
    assert n_attend == 8 and ring.n_valid == sh.n_slots
    big = synth.windowed(steps=synth.WINDOWED_STEPS)
    lo, cnt = big.shape.pos_min[0], big.shape.pos_count[0]
    assert big.shape.n_slots == 5788 and big.shape.n_global == 1246
    for op in big.ops:
        if hasattr(op, "pos"):
            assert op.pos.min() >= lo and op.pos.max() < lo + cnt
