"""Rings in one allocation and the batched position reset against the oracle.

kvring_reset_positions_batch rotates the keys of many rings in one launch
(Runway Characters paper, App. G: every block's window cache is re-rotated
at a reset; §4.1: one allocation holds the caches).  Its result must equal,
bit for bit, the oracle's per-ring reset of every ring: rings at different
fill levels (empty, partly filled, full, wrapped), of different shapes, more
rings than one launch takes, fixed-scale rings, and a reset replayed from a
captured graph."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle.ring import OracleRing
from replay import compare_cache

pytestmark = pytest.mark.gpu


def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_ring_kv_gb300 import kvring as K
    return K, K.load()


def _fill(ring, o, g, counts, t0=0):
    dev = torch.device("cuda")
    sh = ring.heads, ring.head_dim
    for n in counts:
        k = synth.normal_bf16(g, (n, *sh))
        v = synth.normal_bf16(g, (n, *sh))
        pos = synth.lin_pos(t0, n)
        t0 += n
        ring.write(k.to(dev), v.to(dev), torch.from_numpy(pos).to(dev))
        o.write(synth.to_f32(k), synth.to_f32(v), pos)
    return t0


def test_stack_batched_reset_equals_per_ring_resets():
    K, _ = _lib()
    sh = synth.Shape(3, 128, 300, (128,), (-4096,), (8192,))
    stack = K.KVRingStack(5, sh)
    assert stack.workspace.numel() == 5 * stack.stride
    g = synth.rng(82)
    oracles = []
    for i, counts in enumerate(([], [40], [300], [150, 200], [17, 1, 299])):
        o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base)
        _fill(stack.rings[i], o, g, counts)
        oracles.append(o)
    for d in (757, -31):
        stack.reset_positions(d)
        for o in oracles:
            o.reset_positions(d)
        torch.cuda.synchronize()
        for i, (r, o) in enumerate(zip(stack.rings, oracles)):
            assert r.debug_state() == (o.wp, o.n_valid, 0), f"ring {i}"
            compare_cache(r, o, f"ring {i} after the batched reset by {d}")
    stack.close()


def test_batched_reset_of_many_rings_of_different_shapes():
    """45 rings (two launches of at most 32), heads, slots and global slots
    varying; one ring untouched by the batch keeps its keys."""
    K, _ = _lib()
    g = synth.rng(83)
    rings, oracles = [], []
    for i in range(46):
        sh = synth.Shape(1 + i % 3, 64, 40 + 7 * i, (16, 24, 24), (-64, 0, 0), (256, 4, 4), n_global=(i % 4) * 3)
        r = K.KVRing.from_shape(sh)
        o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base, n_global=sh.n_global)
        dev = torch.device("cuda")
        if sh.n_global:
            k = synth.normal_bf16(g, (sh.n_global, sh.heads, 64))
            v = synth.normal_bf16(g, (sh.n_global, sh.heads, 64))
            pos = np.stack([np.full(sh.n_global, -1), np.arange(sh.n_global) % 4, np.zeros(sh.n_global)],
                           1).astype(np.int32)
            r.write_global(k.to(dev), v.to(dev), torch.from_numpy(pos).to(dev))
            o.write_global(synth.to_f32(k), synth.to_f32(v), pos)
        n = (i * 13) % (sh.n_slots - sh.n_global) + 1
        k = synth.normal_bf16(g, (n, sh.heads, 64))
        v = synth.normal_bf16(g, (n, sh.heads, 64))
        pos = np.stack([np.arange(n) % 40, np.arange(n) % 4, (np.arange(n) // 4) % 4], 1).astype(np.int32)
        r.write(k.to(dev), v.to(dev), torch.from_numpy(pos).to(dev))
        o.write(synth.to_f32(k), synth.to_f32(v), pos)
        rings.append(r)
        oracles.append(o)
    K.kvring_reset_positions_batch([r.handle for r in rings[:45]], 5)
    for o in oracles[:45]:
        o.reset_positions(5)
    torch.cuda.synchronize()
    for i, (r, o) in enumerate(zip(rings, oracles)):
        assert r.debug_state() == (o.wp, o.n_valid, 0), f"ring {i}"
        compare_cache(r, o, f"ring {i}")
    for r in rings:
        r.close()


def test_batched_reset_of_calibrated_fixed_scale_rings_and_a_captured_one():
    K, _ = _lib()
    sh = synth.Shape(2, 128, 96, (128,), (-512,), (1024,), scale_mode="static")
    stack = K.KVRingStack(2, sh)
    g = synth.rng(84)
    oracles = [OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base, scale_mode="static")
               for _ in range(2)]
    for r, o in zip(stack.rings, oracles):
        _fill(r, o, g, [50, 30])
        r.calibrate(1.5)
        o.calibrate(1.5)
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        stack.reset_positions(100)
    for rep in range(2):
        graph.replay()
        for o in oracles:
            o.reset_positions(100)
        torch.cuda.synchronize()
        for i, (r, o) in enumerate(zip(stack.rings, oracles)):
            assert r.debug_state() == (o.wp, o.n_valid, 0)
            compare_cache(r, o, f"replay {rep} ring {i}")
    stack.close()


def test_batched_reset_refusals_enqueue_nothing():
    K, lib = _lib()
    a = K.KVRing.from_shape(synth.Shape(1, 64, 32, (64,), (0,), (64,)))
    b = K.KVRing.from_shape(synth.Shape(1, 128, 32, (128,), (0,), (64,)))
    c = K.KVRing.from_shape(synth.Shape(1, 64, 32, (32, 16, 16), (0, 0, 0), (64, 4, 4)))
    s = K.KVRing.from_shape(synth.Shape(1, 64, 32, (64,), (0,), (64,), scale_mode="static"))
    k = torch.ones((4, 1, 64), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((4, 1), dtype=torch.int32, device="cuda")
    for r in (a, s):
        r.write(k, k, pos)

    def call(rs):
        arr = (ctypes.c_void_p * len(rs))(*[r.handle.value for r in rs])
        return lib.kvring_reset_positions_batch(arr, len(rs), 3, None)

    assert call([a, b]) == K.KVRING_ERR_INVALID_ARG         # head_dim differs
    assert call([a, c]) == K.KVRING_ERR_INVALID_ARG         # temporal axis differs
    assert call([a, s]) == K.KVRING_ERR_SEQUENCE            # fixed scales not calibrated
    assert lib.kvring_reset_positions_batch(None, 1, 3, None) == K.KVRING_ERR_INVALID_ARG
    assert call([]) == K.KVRING_ERR_INVALID_ARG
    torch.cuda.synchronize()
    before = a.k_codes.clone()
    assert torch.equal(a.k_codes, before) and a.debug_state() == (4, 4, 0)
    for r in (a, b, c, s):
        r.close()
