"""GPU parity of the RMS norm of Q and K ahead of RoPE (kvring_set_qk_norm)
against oracle/norm.py: the K codes and scales bit for bit, the attention
within the usual tolerance.

Runway Characters paper, §4.4 "Fused pre-attention" and Appendix G.
Collected last, after the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import norm
from oracle.ring import OracleRing
from replay import compare_attention, compare_cache

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _ring(shape):
    from fp8_ring_kv_gb300.kvring import KVRing
    return KVRing.from_shape(shape)


def _weights(g, H, D):
    """bf16 [H, D] norm weights around 1, as a CPU tensor and its float32 values."""
    w = torch.from_numpy((g.standard_normal((H, D)) * 0.3 + 1.0).astype(np.float32)).to(torch.bfloat16)
    return w, synth.to_f32(w)


def test_qk_norm_tiny_with_globals_every_call():
    sh = synth.Shape(2, 64, 58, (16, 24, 24), (-1, 0, 0), (8, 4, 4), n_global=10)
    H, D = sh.heads, sh.head_dim
    g = synth.rng(90)
    wq, wq32 = _weights(g, H, D)
    wk, wk32 = _weights(g, H, D)
    ring = _ring(sh)
    dev = torch.device("cuda")
    wq_d, wk_d = wq.to(dev), wk.to(dev)
    ring.set_qk_norm(wq_d, wk_d, EPS)
    o = OracleRing(H, D, sh.n_slots, sh.axis_dims, sh.rope_base, n_global=sh.n_global)

    def grid(t, n):
        i = np.arange(n)
        return np.stack([np.full(n, t), i // 4 % 4, i % 4], axis=1).astype(np.int32)

    k = synth.normal_bf16(g, (10, H, D)) * 4
    v = synth.normal_bf16(g, (10, H, D))
    ring.write_global(k.to(dev), v.to(dev), torch.from_numpy(grid(-1, 10)).to(dev))
    o.write_global(synth.to_f32(k), synth.to_f32(v), grid(-1, 10), norm_k=(wk32, EPS))
    assert ring.debug_state() == (o.wp, o.n_valid, 0)
    compare_cache(ring, o, "global write with the norm")
    for s in range(6):
        if s == 5:
            ring.reset_positions(5)
            o.reset_positions(5)
            compare_cache(ring, o, "reset")
        n = 16 if s != 2 else 7
        k = synth.normal_bf16(g, (n, H, D)) * 4
        v = synth.normal_bf16(g, (n, H, D))
        q = synth.normal_bf16(g, (n, H, D)) * 4
        pos = grid(s % 6, n)
        ring.write(k.to(dev), v.to(dev), torch.from_numpy(pos).to(dev))
        o.write(synth.to_f32(k), synth.to_f32(v), pos, norm_k=(wk32, EPS))
        assert ring.debug_state() == (o.wp, o.n_valid, 0)
        compare_cache(ring, o, f"write {s} with the norm")
        out = ring.attend(q.to(dev), torch.from_numpy(pos).to(dev)).cpu().numpy()
        compare_attention(out, o.attend(synth.to_f32(q), pos, norm_q=(wq32, EPS)), f"attend {s} with the norm")
    ring.close()


def test_qk_norm_at_the_single_call_shape():
    """24 x 128 heads, a 5,788-token prefill and a 757-token write, 1% of the
    channels x8: every K code and scale; the attention on three heads."""
    wl = synth.single()
    sh = wl.shape
    H, D = sh.heads, sh.head_dim
    g = synth.rng(91)
    wq, wq32 = _weights(g, H, D)
    wk, wk32 = _weights(g, H, D)
    dev = torch.device("cuda")
    ring = _ring(sh)
    wq_d, wk_d = wq.to(dev), wk.to(dev)
    ring.set_qk_norm(wq_d, wk_d, EPS)
    o = OracleRing(H, D, sh.n_slots, sh.axis_dims, sh.rope_base)
    for op in wl.ops:
        if isinstance(op, synth.Write):
            ring.write(op.k.to(dev), op.v.to(dev), torch.from_numpy(op.pos).to(dev))
            o.write(synth.to_f32(op.k), synth.to_f32(op.v), op.pos, norm_k=(wk32, EPS))
            assert ring.debug_state() == (o.wp, o.n_valid, 0)
        else:
            out = ring.attend(op.q.to(dev), torch.from_numpy(op.pos).to(dev)).cpu().numpy()
            compare_cache(ring, o, "single call with the norm")
            heads = [0, 11, 23]
            ref = o.attend(synth.to_f32(op.q), op.pos, heads=heads, norm_q=(wq32, EPS))
            compare_attention(out[:, heads], ref, "attend with the norm")
    ring.close()


def test_qk_norm_host_rules_and_switching_off():
    from fp8_ring_kv_gb300 import kvring as K
    lib = K.load()
    sh = synth.Shape(2, 64, 32, (64,), (0,), (64,))
    H, D = sh.heads, sh.head_dim
    g = synth.rng(92)
    w, w32 = _weights(g, H, D)
    dev = torch.device("cuda")
    wd = w.to(dev)
    ring = _ring(sh)
    h = ring.handle
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)  # noqa: E731
    assert lib.kvring_set_qk_norm(h, p(wd), p(wd), 0.0) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_set_qk_norm(h, p(wd), p(wd), float("inf")) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_set_qk_norm(h, p(wd, 2), None, 1e-6) == K.KVRING_ERR_MISALIGNED
    o = OracleRing(H, D, sh.n_slots, sh.axis_dims, sh.rope_base)
    k = synth.normal_bf16(g, (8, H, D)) * 4
    v = synth.normal_bf16(g, (8, H, D))
    pos = synth.lin_pos(0, 8)
    ring.set_qk_norm(None, wd, EPS)                       # K only
    ring.write(k.to(dev), v.to(dev), torch.from_numpy(pos).to(dev))
    o.write(synth.to_f32(k), synth.to_f32(v), pos, norm_k=(w32, EPS))
    ring.set_qk_norm(None, None)                          # off again
    ring.write(k.to(dev), v.to(dev), torch.from_numpy(pos + 8).to(dev))
    o.write(synth.to_f32(k), synth.to_f32(v), pos + 8)
    torch.cuda.synchronize()
    compare_cache(ring, o, "norm on, then off")
    q = synth.normal_bf16(g, (5, H, D))
    qp = synth.lin_pos(10, 5)
    out = ring.attend(q.to(dev), torch.from_numpy(qp).to(dev)).cpu().numpy()
    compare_attention(out, o.attend(synth.to_f32(q), qp), "attend without a Q norm")
    ring.close()
