"""kvring_attend_noalloc against kvring_attend (collected last on purpose: it
must also pass after every other test has run in the same process).

The two calls run the same kernels; only where the per-call query scratch
lives differs (a fixed device array inside the library instead of the ring's
workspace).  Two calls in a row, with different query counts and queries,
must each agree with kvring_attend within the attention tolerance, leave the
ring unchanged, and allocate no device memory."""
import numpy as np
import pytest
import torch

import synth
from replay import ATT_MAX_ABS, ATT_MEAN_ABS

pytestmark = pytest.mark.gpu


def _filled_ring():
    from fp8_ring_kv_gb300.kvring import KVRing
    wl = synth.single()
    ring = KVRing.from_shape(wl.shape)
    dev = torch.device("cuda")
    for op in wl.ops:
        if isinstance(op, synth.Write):
            ring.write(op.k.to(dev), op.v.to(dev), torch.from_numpy(op.pos).to(dev))
    return wl.shape, ring


def _queries(shape, n_q, seed):
    g = synth.rng(90, seed)
    q = synth.normal_bf16(g, (n_q, shape.heads, shape.head_dim)).cuda()
    # positions inside the RoPE table: pos_min .. pos_min + pos_count - 1
    start = min(shape.n_slots + 16 * seed, shape.pos_min[0] + shape.pos_count[0] - n_q)
    pos = torch.from_numpy(synth.lin_pos(start, n_q)).cuda()
    return q, pos


def _close(a, b, what):
    err = (a.double() - b.double()).abs()
    assert torch.isfinite(a).all(), f"{what}: non-finite output"
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= ATT_MAX_ABS and mean <= ATT_MEAN_ABS, f"{what}: max {mx:.3e} mean {mean:.3e}"


def test_noalloc_matches_attend_on_two_calls_in_a_row():
    from fp8_ring_kv_gb300 import kvring as K
    shape, ring = _filled_ring()
    torch.cuda.synchronize()
    state0 = ring.debug_state()
    calls = []
    for i, n_q in enumerate((synth.NEW_TOKENS, 300)):
        q, pos = _queries(shape, n_q, i)
        want = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        got = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        calls.append((q, pos, want, got))
    # warm the ordinary path and the no-alloc set-up before the memory check
    q, pos, want, got = calls[0]
    K.kvring_attend(ring.handle, q, pos, q.shape[0], want)
    K.kvring_attend_noalloc(ring.handle, q, pos, q.shape[0], got)
    torch.cuda.synchronize()
    # no-alloc calls alone leave the ring's whole workspace as it was (its
    # query scratch included)
    before = ring.workspace.clone()
    for q, pos, want, got in calls:
        K.kvring_attend_noalloc(ring.handle, q, pos, q.shape[0], got)
    torch.cuda.synchronize()
    assert torch.equal(ring.workspace, before), "kvring_attend_noalloc wrote into the ring's workspace"
    del before
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for i, (q, pos, want, got) in enumerate(calls):
        K.kvring_attend_noalloc(ring.handle, q, pos, q.shape[0], got)
        K.kvring_attend(ring.handle, q, pos, q.shape[0], want)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device memory changed by {free0 - free1} bytes"
    for i, (q, pos, want, got) in enumerate(calls):
        _close(got, want, f"call {i} (n_q {q.shape[0]})")
    assert ring.debug_state() == state0
    ring.close()


def test_noalloc_rejects_requests_beyond_the_static_scratch():
    from fp8_ring_kv_gb300 import kvring as K
    shape, ring = _filled_ring()
    H, D = shape.heads, shape.head_dim

    def need(n):
        ru = lambda x, a: (x + a - 1) // a * a  # noqa: E731
        return ru(n * H * D, 1024) + H * ru(n, 4) * 4 + 2 * H * 4

    n_max = max(n for n in range(1, 8192) if need(n) <= K.KVRING_NOALLOC_SCRATCH_BYTES)
    q, pos = _queries(shape, n_max + 1, 7)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(K.KVRingError, match="static scratch"):
        K.kvring_attend_noalloc(ring.handle, q, pos, n_max + 1, out)
    # the largest request that fits runs and agrees with kvring_attend
    want = torch.empty_like(out)
    got = torch.empty_like(out)
    big = K.KVRing.from_shape(shape, max_queries=n_max)
    for op in synth.single().ops:
        if isinstance(op, synth.Write):
            big.write(op.k.cuda(), op.v.cuda(), torch.from_numpy(op.pos).cuda())
    K.kvring_attend_noalloc(big.handle, q, pos, n_max, got)
    K.kvring_attend(big.handle, q, pos, n_max, want)
    torch.cuda.synchronize()
    _close(got[:n_max], want[:n_max], f"n_q {n_max}")
    assert big.debug_state()[2] == 0 and ring.debug_state()[2] == 0
    big.close()
    ring.close()
