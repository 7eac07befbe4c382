"""Replay a synthetic workload on the CUDA library and on the oracle, side by side.

The library is driven through its C ABI (``fp8_ring_kv_gb300.kvring``); the
oracle keeps its own FP8 cache from the same bf16 inputs.  After every call
the two are compared:

* ring state (write position, valid count): exact;
* K/V e4m3 codes and fp32 scales: bit for bit (both sides take the e4m3
  decision in fp32 from identical fp32 inputs, so the codes must agree);
* attention: max |out - oracle| <= ATT_MAX_ABS and mean <= ATT_MEAN_ABS.
"""
import time
from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from oracle.ring import OracleRing

ATT_MAX_ABS = 1e-2
ATT_MEAN_ABS = 1e-3


@dataclass
class Report:
    writes: int = 0
    resets: int = 0
    attends: int = 0
    attend_checked: int = 0
    worst_max_abs: float = 0.0
    worst_mean_abs: float = 0.0
    attend_stats: list = field(default_factory=list)
    seconds: float = 0.0


def gpu_ring(shape, out_f32=True):
    from fp8_ring_kv_gb300.kvring import KVRing, KVRING_OUT_F32, KVRING_OUT_BF16
    return KVRing.from_shape(shape, KVRING_OUT_F32 if out_f32 else KVRING_OUT_BF16)


def compare_cache(g, o: OracleRing, what=""):
    """Bit-exact comparison of the library's cache with the oracle's."""
    S = o.S
    kc = g.k_codes.cpu().numpy()
    vc = g.v_codes.cpu().numpy()
    ks = g.k_scales[:, :S].cpu().numpy()
    vs = g.v_scales[:, :S].cpu().numpy()
    n = o.n_valid
    for name, got, want in (("k_codes", kc[:, :n], o.k_codes[:, :n]), ("v_codes", vc[:, :n], o.v_codes[:, :n])):
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{what}: {name} differ at {len(bad)} places, first {bad[:5].tolist()}"
    for name, got, want in (("k_scale", ks[:, :n], o.k_scale[:, :n]), ("v_scale", vs[:, :n], o.v_scale[:, :n])):
        bad = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, f"{what}: {name} differ at {len(bad)} places, first {bad[:5].tolist()}"


def compare_attention(out, ref, what="", allowance=None):
    err = np.abs(out.astype(np.float64) - ref)
    if allowance is not None:
        err = np.maximum(err - allowance, 0.0)
    mx, mean = float(err.max()), float(err.mean())
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    assert mx <= ATT_MAX_ABS and mean <= ATT_MEAN_ABS, f"{what}: max|err| {mx:.3e} mean|err| {mean:.3e}"
    return mx, mean


def replay(wl: synth.Workload, *, cache_every=1, attend_filter=None, oracle_rings=None, attend_heads=None,
           out_f32=True, stream=None) -> Report:
    """Run ``wl`` on the GPU and the oracle.

    cache_every    compare the whole cache after every n-th write/reset (0: never)
    attend_filter  tag -> bool: which attends the oracle recomputes (all by default)
    oracle_rings   which rings the oracle follows (all by default)
    attend_heads   heads the oracle recomputes per checked attend (all by default)
    """
    t0 = time.time()
    sh = wl.shape
    rings = [gpu_ring(sh, out_f32) for _ in range(wl.n_rings)]
    follow = set(range(wl.n_rings)) if oracle_rings is None else set(oracle_rings)
    refs = {r: OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base, n_global=sh.n_global,
                          scale_mode=sh.scale_mode)
            for r in follow}
    rep = Report()
    n_cache = 0
    dev = torch.device("cuda")
    for op in wl.ops:
        g = rings[op.ring]
        o = refs.get(op.ring)
        if isinstance(op, (synth.Write, synth.WriteGlobal)):
            glob = isinstance(op, synth.WriteGlobal)
            (g.write_global if glob else g.write)(op.k.to(dev), op.v.to(dev), torch.from_numpy(op.pos).to(dev))
            rep.writes += 1
            if o is not None:
                (o.write_global if glob else o.write)(synth.to_f32(op.k), synth.to_f32(op.v), op.pos)
                wp, nv, err = g.debug_state()
                assert (wp, nv, err) == (o.wp, o.n_valid, 0), f"state {(wp, nv, err)} vs {(o.wp, o.n_valid)}"
                n_cache += 1
                if cache_every and n_cache % cache_every == 0:
                    compare_cache(g, o, f"after write {rep.writes}")
        elif isinstance(op, synth.Calibrate):
            g.calibrate(op.margin)
            if o is not None:
                o.calibrate(op.margin)
                assert g.debug_state() == (o.wp, o.n_valid, 0)
                compare_cache(g, o, "after the calibration")
        elif isinstance(op, synth.Reset):
            g.reset_positions(op.d)
            rep.resets += 1
            if o is not None:
                o.reset_positions(op.d)
                n_cache += 1
                if cache_every:
                    compare_cache(g, o, f"after reset {rep.resets}")
        else:
            out = g.attend(op.q.to(dev), torch.from_numpy(op.pos).to(dev))
            rep.attends += 1
            if o is None or (attend_filter is not None and not attend_filter(op.tag)):
                continue
            heads = None if attend_heads is None else list(attend_heads)
            ref = o.attend(synth.to_f32(op.q), op.pos, heads=heads)
            got = out.float().cpu().numpy()
            if heads is not None:
                got = got[:, heads]
            # bf16 output: half a bf16 ulp of the value on top of the tolerance
            allow = None if out_f32 else np.abs(ref) * 2.0 ** -8
            mx, mean = compare_attention(got, ref, f"attend {op.tag} ring {op.ring}", allow)
            rep.attend_checked += 1
            rep.worst_max_abs = max(rep.worst_max_abs, mx)
            rep.worst_mean_abs = max(rep.worst_mean_abs, mean)
            rep.attend_stats.append((op.ring, op.tag, mx, mean))
    torch.cuda.synchronize()
    for g in rings:
        wp, nv, err = g.debug_state()
        assert err == 0, f"device error word {err}"
        g.close()
    rep.seconds = time.time() - t0
    return rep
