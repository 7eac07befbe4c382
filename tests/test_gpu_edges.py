"""Edge cases of the CUDA path against the oracle and the C ABI's error
contract: the write kernel's quantiser on raw rows, host-side rejections
with a live ring, an empty ring, positions outside the RoPE table, and a
write of a whole ring's worth of tokens."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import quant
from oracle.ring import OracleRing
from replay import compare_attention, compare_cache

pytestmark = pytest.mark.gpu


def _lib():
    from fp8_ring_kv_gb300 import kvring as K
    return K, K.load()


@pytest.mark.parametrize("d", [16, 32, 64, 128, 256])
def test_debug_quantize_bit_exact(d):
    """kvring_debug_quantize (the write kernel's quantiser) on fp32 rows:
    codes and scales bit for bit equal to the oracle's quantize_rows."""
    K, _ = _lib()
    g = np.random.default_rng(d)
    rows = 3000
    x = (g.standard_normal((rows, d)) * np.exp2(g.uniform(-30, 30, (rows, 1)))).astype(np.float32)
    x[0] = 0.0                                   # zero row
    x[1, :] = -0.0
    x[1, 3] = -1e-30                             # tiny magnitudes
    x[2, 5] = 448.0                              # amax exactly 448
    x[3] = np.float32(2.0 ** -140)               # subnormal fp32
    x[4, ::2] *= -1
    xd = torch.from_numpy(x).cuda()
    codes = torch.empty((rows, d), dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    K.kvring_debug_quantize(xd, rows, d, codes, scales)
    torch.cuda.synchronize()
    with np.errstate(over="ignore"):   # 448 / amax overflows to inf on the subnormal row, as in fp32
        want_c, want_s = quant.quantize_rows(x)
    got_c, got_s = codes.cpu().numpy(), scales.cpu().numpy()
    bad = np.argwhere(got_c != want_c)
    assert bad.size == 0, f"codes differ at {len(bad)} places, first {bad[:5].tolist()}"
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32))


def _ring(shape, **kw):
    from fp8_ring_kv_gb300.kvring import KVRing
    return KVRing.from_shape(shape, **kw)


def _tiny_shape(n_slots=64, pos_count=256):
    return synth.Shape(2, 64, n_slots, (64,), (0,), (pos_count,))


def test_host_rejections_with_a_live_ring():
    K, lib = _lib()
    sh = _tiny_shape()
    ring = _ring(sh, max_queries=32)
    dev = torch.device("cuda")
    k = torch.zeros((sh.n_slots + 1, sh.heads, sh.head_dim), dtype=torch.bfloat16, device=dev)
    pos = torch.zeros((sh.n_slots + 1, 1), dtype=torch.int32, device=dev)
    h = ring.handle
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)  # noqa: E731
    # more tokens than slots, zero tokens, misaligned inputs
    assert lib.kvring_write(h, p(k), p(k), p(pos), sh.n_slots + 1, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_write(h, p(k), p(k), p(pos), 0, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_write(h, p(k, 2), p(k), p(pos), 4, None) == K.KVRING_ERR_MISALIGNED
    assert lib.kvring_write(h, p(k), p(k), p(pos, 2), 4, None) == K.KVRING_ERR_MISALIGNED
    # more queries than the workspace's scratch holds
    out = torch.empty((33, sh.heads, sh.head_dim), dtype=torch.float32, device=dev)
    q = torch.zeros((33, sh.heads, sh.head_dim), dtype=torch.bfloat16, device=dev)
    assert lib.kvring_attend(h, p(q), p(pos), 33, p(out), None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_attend(h, p(q), p(pos), 0, p(out), None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_attend(h, p(q), p(pos), 4, p(out, 4), None) == K.KVRING_ERR_MISALIGNED
    torch.cuda.synchronize()
    # nothing was enqueued: the ring is still empty and clean
    assert ring.debug_state() == (0, 0, 0)
    ring.close()


def test_attend_on_an_empty_ring_gives_zeros_and_a_flag():
    K, _ = _lib()
    sh = _tiny_shape()
    ring = _ring(sh)
    q = torch.ones((5, sh.heads, sh.head_dim), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((5, 1), dtype=torch.int32, device="cuda")
    out = ring.attend(q, pos)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    wp, nv, err = ring.debug_state()
    assert (wp, nv) == (0, 0) and err & K.KVRING_DEVERR_EMPTY
    ring.close()


def test_positions_outside_the_table_are_clamped_and_flagged():
    K, _ = _lib()
    sh = _tiny_shape(pos_count=16)
    ring = _ring(sh)
    g = synth.rng(77)
    n = 8
    k = synth.normal_bf16(g, (n, sh.heads, sh.head_dim))
    v = synth.normal_bf16(g, (n, sh.heads, sh.head_dim))
    pos = np.array([[-3], [0], [5], [15], [16], [40], [7], [2]], dtype=np.int32)
    ring.write(k.cuda(), v.cuda(), torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    wp, nv, err = ring.debug_state()
    assert (wp, nv) == (n, n) and err & K.KVRING_DEVERR_POS_RANGE
    # the clamped positions are the table's ends
    o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base)
    o.write(synth.to_f32(k), synth.to_f32(v), np.clip(pos, 0, 15))
    compare_cache(ring, o, "clamped write")
    ring.close()


def test_write_of_a_whole_ring_then_wrapping_writes():
    """n_new == S fills every slot in one call; later writes wrap around."""
    sh = synth.Shape(3, 128, 200, (32, 48, 48), (0, 0, 0), (1024, 16, 16))
    ring = _ring(sh)
    o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base)
    g = synth.rng(78)
    dev = torch.device("cuda")
    t0 = 0
    for n in (200, 77, 150, 200, 1):
        k = synth.normal_bf16(g, (n, sh.heads, sh.head_dim))
        v = synth.normal_bf16(g, (n, sh.heads, sh.head_dim))
        pos = np.stack([t0 + np.arange(n), np.arange(n) % 16, (np.arange(n) // 16) % 16], 1).astype(np.int32)
        t0 += n
        ring.write(k.to(dev), v.to(dev), torch.from_numpy(pos).to(dev))
        o.write(synth.to_f32(k), synth.to_f32(v), pos)
        assert ring.debug_state() == (o.wp, o.n_valid, 0)
        compare_cache(ring, o, f"after writing {n}")
    q = synth.normal_bf16(g, (130, sh.heads, sh.head_dim))
    qpos = np.stack([t0 + np.arange(130), np.arange(130) % 16, np.zeros(130)], 1).astype(np.int32)
    out = ring.attend(q.to(dev), torch.from_numpy(qpos).to(dev)).cpu().numpy()
    compare_attention(out, o.attend(synth.to_f32(q), qpos), "attend after wraps")
    ring.close()


def test_global_slot_call_order_is_checked_on_the_host():
    """kvring_write_global: exactly n_global tokens, once, before any window
    write; window writes carry at most n_slots - n_global tokens.  Rejected
    calls enqueue nothing."""
    K, lib = _lib()
    sh = synth.Shape(2, 64, 40, (64,), (0,), (256,), n_global=8)
    ring = _ring(sh)
    dev = torch.device("cuda")
    k = torch.zeros((40, sh.heads, sh.head_dim), dtype=torch.bfloat16, device=dev)
    pos = torch.zeros((40, 1), dtype=torch.int32, device=dev)
    h = ring.handle
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.kvring_write(h, p(k), p(k), p(pos), 4, None) == K.KVRING_ERR_SEQUENCE
    assert lib.kvring_write_global(h, p(k), p(k), p(pos), 7, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_write_global(h, p(k), p(k), p(pos), 9, None) == K.KVRING_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert ring.debug_state() == (0, 0, 0)
    assert lib.kvring_write_global(h, p(k), p(k), p(pos), 8, None) == K.KVRING_OK
    assert lib.kvring_write_global(h, p(k), p(k), p(pos), 8, None) == K.KVRING_ERR_SEQUENCE
    assert lib.kvring_write(h, p(k), p(k), p(pos), 33, None) == K.KVRING_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert ring.debug_state() == (0, 8, 0)
    assert lib.kvring_write(h, p(k), p(k), p(pos), 32, None) == K.KVRING_OK
    torch.cuda.synchronize()
    assert ring.debug_state() == (0, 40, 0)
    ring.close()
    plain = _ring(_tiny_shape())
    assert lib.kvring_write_global(plain.handle, p(k), p(k), p(pos), 1, None) == K.KVRING_ERR_INVALID_ARG
    plain.close()


def test_reset_before_any_window_write_leaves_the_globals():
    """A reset with only the globals written rotates nothing."""
    sh = synth.Shape(2, 64, 40, (16, 24, 24), (-8, 0, 0), (16, 4, 4), n_global=8)
    ring = _ring(sh)
    o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base, n_global=8)
    g = synth.rng(79)
    k = synth.normal_bf16(g, (8, sh.heads, sh.head_dim))
    v = synth.normal_bf16(g, (8, sh.heads, sh.head_dim))
    pos = np.stack([np.full(8, -1), np.arange(8) // 4, np.arange(8) % 4], 1).astype(np.int32)
    ring.write_global(k.cuda(), v.cuda(), torch.from_numpy(pos).cuda())
    o.write_global(synth.to_f32(k), synth.to_f32(v), pos)
    ring.reset_positions(5)
    o.reset_positions(5)
    assert ring.debug_state() == (0, 8, 0)
    compare_cache(ring, o, "globals after a reset")
    q = synth.normal_bf16(g, (5, sh.heads, sh.head_dim))
    qpos = np.stack([np.arange(5), np.zeros(5), np.zeros(5)], 1).astype(np.int32)
    out = ring.attend(q.cuda(), torch.from_numpy(qpos).cuda()).cpu().numpy()
    compare_attention(out, o.attend(synth.to_f32(q), qpos), "attend over the globals alone")
    ring.close()


def test_calibration_call_rules():
    K, lib = _lib()
    sh = synth.Shape(2, 64, 40, (64,), (0,), (256,), scale_mode="static")
    ring = _ring(sh)
    dev = torch.device("cuda")
    k = torch.ones((4, sh.heads, sh.head_dim), dtype=torch.bfloat16, device=dev)
    pos = torch.zeros((4, 1), dtype=torch.int32, device=dev)
    h = ring.handle
    assert lib.kvring_calibrate(h, 1.5, None) == K.KVRING_ERR_SEQUENCE          # nothing written yet
    ring.write(k, k, pos)
    assert lib.kvring_reset_positions(h, 3, None) == K.KVRING_ERR_SEQUENCE      # calibrate first
    assert lib.kvring_calibrate(h, 0.0, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_calibrate(h, float("nan"), None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_calibrate(h, 1.5, None) == K.KVRING_OK
    assert lib.kvring_calibrate(h, 1.5, None) == K.KVRING_ERR_SEQUENCE          # once
    assert lib.kvring_reset_positions(h, 3, None) == K.KVRING_OK
    # the fixed K scales were taken from un-normalised keys: the K norm may
    # not change any more, the Q norm may
    w = torch.ones((sh.heads, sh.head_dim), dtype=torch.bfloat16, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.kvring_set_qk_norm(h, None, p(w), 1e-6) == K.KVRING_ERR_SEQUENCE
    assert lib.kvring_set_qk_norm(h, p(w), None, 1e-6) == K.KVRING_OK
    torch.cuda.synchronize()
    assert ring.debug_state() == (4, 4, 0)
    ring.close()
    plain = _ring(_tiny_shape())
    plain.write(k, k, pos)
    assert lib.kvring_calibrate(plain.handle, 1.5, None) == K.KVRING_ERR_SEQUENCE  # per-token scales
    plain.close()


def test_a_captured_write_follows_the_calibration():
    """The scale mode is read on the device: one captured write, replayed
    before and after the calibration, quantises per token and then with the
    fixed scales."""
    sh = synth.Shape(2, 64, 64, (16, 24, 24), (0, 0, 0), (8, 4, 4), scale_mode="static")
    ring = _ring(sh)
    o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base, scale_mode="static")
    g = synth.rng(80)
    k = synth.normal_bf16(g, (12, sh.heads, sh.head_dim))
    v = synth.normal_bf16(g, (12, sh.heads, sh.head_dim))
    pos = np.stack([np.arange(12) % 8, np.arange(12) % 4, np.arange(12) // 4 % 4], 1).astype(np.int32)
    kd, vd, pd = k.cuda(), v.cuda(), torch.from_numpy(pos).cuda()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ring.write(kd, vd, pd)
    torch.cuda.synchronize()
    assert ring.debug_state() == (0, 0, 0)          # captured, not run
    graph.replay()
    o.write(synth.to_f32(k), synth.to_f32(v), pos)
    ring.calibrate(1.5)
    o.calibrate(1.5)
    graph.replay()
    o.write(synth.to_f32(k), synth.to_f32(v), pos)
    torch.cuda.synchronize()
    assert ring.debug_state() == (o.wp, o.n_valid, 0)
    compare_cache(ring, o, "captured write after the calibration")
    ring.close()


def test_fewer_queries_than_the_previous_call():
    """The query scratch keeps the rows of an earlier, larger call; a later
    call with fewer queries (a partial last query tile) must not be affected
    by them.  757, then 300, then 5 queries on one ring, each against the
    oracle."""
    wl = synth.single()
    ops = list(wl.ops)
    sh = wl.shape
    ring = _ring(sh)
    o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base)
    dev = torch.device("cuda")
    for op in ops:
        if isinstance(op, synth.Write):
            ring.write(op.k.to(dev), op.v.to(dev), torch.from_numpy(op.pos).to(dev))
            o.write(synth.to_f32(op.k), synth.to_f32(op.v), op.pos)
    g = synth.rng(81)
    heads = [0, 7, 23]
    for n_q in (757, 300, 5):
        q = synth.normal_bf16(g, (n_q, sh.heads, sh.head_dim))
        qpos = synth.lin_pos(sh.n_slots, n_q)
        out = ring.attend(q.to(dev), torch.from_numpy(qpos).to(dev)).cpu().numpy()[:, heads]
        compare_attention(out, o.attend(synth.to_f32(q), qpos, heads=heads), f"{n_q} queries")
    assert ring.debug_state()[2] == 0
    ring.close()


def test_a_wait_that_runs_out_returns_an_error_status():
    """The kernels' bounded barrier wait, on a barrier that never completes:
    after its limit the block records KVRING_DEVERR_TIMEOUT and returns, and
    the device keeps working (the same wait that completes reports 0)."""
    K, _ = _lib()
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    limit = 20_000_000                                   # 20 ms
    K.kvring_debug_wait_timeout(limit, False, out)
    torch.cuda.synchronize()
    err, ns = out.tolist()
    assert err == K.KVRING_DEVERR_TIMEOUT and ns >= limit
    K.kvring_debug_wait_timeout(limit, True, out)
    torch.cuda.synchronize()
    err, ns = out.tolist()
    assert err == 0 and ns < limit
    assert int((torch.arange(8, device="cuda") * 2).sum()) == 56
