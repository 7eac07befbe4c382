"""Seeded synthetic workloads shared by the tests, the benchmark and the oracle.

This module holds no arithmetic of the method (no RoPE, no quantisation, no
attention): it only draws bf16 inputs from seeded generators and lays out the
sequence of calls and the integer positions of each workload.

Inputs are i.i.d. N(0, 1) drawn in float32 by numpy's PCG64 generator and
rounded to bfloat16 (round to nearest even).  The paper's own K/V/Q come from a
57B video model on live speech and are not available; these normal draws, with
1% of the channels scaled by 8 where a workload says so, stand in for them.

Workloads (the shapes the paper describes: 757 new tokens per write into a
5,788-slot cache, 24 heads of 128 per tensor-parallel slice):

1. ``tiny``      H=1, D=64, S=64, N=16, six writes (the ring wraps), reset by
                 d=32 after the 4th write, an attend after every write.
2. ``single``    H=24, D=128, S=5,788: one prefill write of 5,788 tokens, then
                 one write of 757 and one attend of 757 queries; 1% of the
                 channels x8.
3. ``sustained`` H=24, D=128, S=5,788: 84 steps of write(757)+attend(757),
                 positions advance 757 per step and are reset by 42*757 before
                 step 42 and after step 83 (followed by one more attend).
4. ``chunk``     60 rings (layers) x 8 chunks; per chunk one write of 757 and 4
                 attends (denoising passes) per ring; reset by 4*757 before
                 chunk 4.
5. ``sweep``     H in {8,24,48} x D in {64,128} x S in {1447,2894,5788,11576},
                 N = round(S*757/5788), 3-axis (t,h,w) positions on a latent
                 grid with aspect 1088:704.
6. ``windowed``  the paper's own layout: 1,246 global slots written once (at
                 temporal positions -1246 .. -1), then a window ring of six
                 757-token frames; ten steps of write(757)+attend(757) at
                 (s mod 7)*757 + i, the window reset by 7*757 before step 7;
                 1% of the channels x8.  ``windowed_tiny``: the same on
                 H=2, D=64, 10 globals, three 16-token frames, 3-axis RoPE.
7. ``static_scales`` / ``static_scales_tiny``: the windowed workloads (ten
                 steps, the reset before step 7) on a ring with per-head
                 fixed scales, calibrated (margin 1.5) on entering the
                 seventh step; in the tiny one step 8's K and V are scaled x3
                 so that values pass the calibrated range.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from functools import lru_cache
from typing import Iterator, List, Optional, Tuple

import numpy as np
import torch

NEW_TOKENS = 757
SLOTS = 5788


# ---------------------------------------------------------------------------
# shapes and calls
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Shape:
    heads: int
    head_dim: int
    n_slots: int
    axis_dims: Tuple[int, ...]
    pos_min: Tuple[int, ...]        # RoPE table coverage per axis: positions
    pos_count: Tuple[int, ...]      #   pos_min .. pos_min + pos_count - 1
    rope_base: float = 10000.0
    n_global: int = 0               # global slots ahead of the window ring
    scale_mode: str = "token"       # "token" or "static" (per-head scales fixed by a calibration)

    @property
    def n_axes(self):
        return len(self.axis_dims)


@dataclass
class Write:
    k: torch.Tensor            # bf16 [N, H, D] (CPU)
    v: torch.Tensor
    pos: np.ndarray            # int32 [N, n_axes]
    ring: int = 0


@dataclass
class WriteGlobal:
    k: torch.Tensor            # bf16 [n_global, H, D] (CPU)
    v: torch.Tensor
    pos: np.ndarray            # int32 [n_global, n_axes]
    ring: int = 0


@dataclass
class Calibrate:
    margin: float = 1.5
    ring: int = 0


@dataclass
class Reset:
    d: int
    ring: int = 0


@dataclass
class Attend:
    q: torch.Tensor            # bf16 [Nq, H, D]
    pos: np.ndarray            # int32 [Nq, n_axes]
    ring: int = 0
    tag: str = ""


@dataclass
class Workload:
    name: str
    shape: Shape
    n_rings: int
    ops: Iterator           # of WriteGlobal / Write / Calibrate / Reset / Attend
    note: str = ""


# ---------------------------------------------------------------------------
# draws
# ---------------------------------------------------------------------------
def rng(*seed) -> np.random.Generator:
    return np.random.default_rng(list(seed) if len(seed) > 1 else seed[0])


def normal_bf16(g: np.random.Generator, shape, scale_channels: Optional[np.ndarray] = None):
    """N(0,1) float32 draws rounded to bf16.  ``scale_channels``: flat indices
    h*D + d of the channels multiplied by 8 (exact in bf16)."""
    x = g.standard_normal(size=shape, dtype=np.float32)
    if scale_channels is not None and len(scale_channels):
        flat = x.reshape(shape[0], -1)
        flat[:, scale_channels] *= np.float32(8.0)
    return torch.from_numpy(x).to(torch.bfloat16)


def outlier_channels(g: np.random.Generator, heads: int, head_dim: int, frac=0.01):
    n = int(math.floor(frac * heads * head_dim + 0.5))
    return np.sort(g.permutation(heads * head_dim)[:n])


def to_f32(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> float32 numpy array (exact)."""
    return t.float().numpy()


def lin_pos(start: int, n: int) -> np.ndarray:
    return (start + np.arange(n, dtype=np.int64)).astype(np.int32).reshape(n, 1)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def tiny() -> Workload:
    H, D, S, N = 1, 64, 64, 16
    shape = Shape(H, D, S, (D,), (0,), (64,))

    def ops():
        g = rng(0)
        for w in range(1, 7):                      # writes are numbered from 1
            start = (w - 1) * N if w <= 4 else (w - 1) * N - 32
            pos = lin_pos(start, N)
            k = normal_bf16(g, (N, H, D))
            v = normal_bf16(g, (N, H, D))
            q = normal_bf16(g, (N, H, D))
            yield Write(k, v, pos)
            yield Attend(q, pos, tag=f"w{w}")
            if w == 4:
                yield Reset(32)
    return Workload("tiny", shape, 1, ops())


def single(n_new: int = NEW_TOKENS) -> Workload:
    H, D, S = 24, 128, SLOTS
    shape = Shape(H, D, S, (D,), (0,), (8192,))

    def ops():
        g = rng(1)
        ch = outlier_channels(g, H, D)
        k = normal_bf16(g, (S, H, D), ch)
        v = normal_bf16(g, (S, H, D), ch)
        yield Write(k, v, lin_pos(0, S))
        k = normal_bf16(g, (n_new, H, D), ch)
        v = normal_bf16(g, (n_new, H, D), ch)
        q = normal_bf16(g, (n_new, H, D), ch)
        pos = lin_pos(S, n_new)
        yield Write(k, v, pos)
        yield Attend(q, pos, tag="call")
    return Workload("single", shape, 1, ops())


SUSTAINED_STEPS = 84
RESET_PERIOD = 42


def sustained(steps: int = SUSTAINED_STEPS) -> Workload:
    H, D, S, N = 24, 128, SLOTS, NEW_TOKENS
    dshift = RESET_PERIOD * N
    shape = Shape(H, D, S, (D,), (-N,), (dshift + N,))

    def ops():
        g = rng(2)
        q = pos = None
        for s in range(steps):
            if s > 0 and s % RESET_PERIOD == 0:
                yield Reset(dshift)
            pos = lin_pos((s % RESET_PERIOD) * N, N)
            k = normal_bf16(g, (N, H, D))
            v = normal_bf16(g, (N, H, D))
            q = normal_bf16(g, (N, H, D))
            yield Write(k, v, pos)
            yield Attend(q, pos, tag=f"s{s}")
        if steps % RESET_PERIOD == 0:
            yield Reset(dshift)
            yield Attend(q, (pos.astype(np.int64) - dshift).astype(np.int32), tag="after_reset")
    return Workload("sustained", shape, 1, ops())


CHUNK_LAYERS = 60
CHUNK_PASSES = 4
CHUNKS = 8
_POOL_BLOCKS = 64


@lru_cache(maxsize=1)
def chunk_pool() -> torch.Tensor:
    """64 blocks of [757, 24, 128] bf16 N(0,1) (seed 3).  Each ring draws its
    inputs from this pool through its own seeded permutation, so every input
    inside one ring is a distinct draw."""
    g = rng(3)
    return normal_bf16(g, (_POOL_BLOCKS * NEW_TOKENS, 24, 128)).view(
        _POOL_BLOCKS, NEW_TOKENS, 24, 128)


def chunk_layer_blocks(layer: int) -> np.ndarray:
    return rng(3, layer).permutation(_POOL_BLOCKS)


def chunk(layers: int = CHUNK_LAYERS, chunks: int = CHUNKS, passes: int = CHUNK_PASSES) -> Workload:
    """Ring r = layer.  Per ring: prefill S tokens at positions -S..-1; chunk c
    writes 757 tokens at c*757 + i (c < 4) or (c-4)*757 + i (c >= 4, after the
    reset by 4*757 before chunk 4) and attends 4 query sets at those positions."""
    H, D, S, N = 24, 128, SLOTS, NEW_TOKENS
    if not (1 <= passes <= 4 and 1 <= chunks <= CHUNKS):
        raise ValueError("at most 8 chunks of 4 passes")
    shape = Shape(H, D, S, (D,), (-S,), (S + 4 * N,))
    pool = chunk_pool()

    def block(i):
        return pool[int(i)]

    def ops():
        perms = [chunk_layer_blocks(l) for l in range(layers)]
        for l in range(layers):
            kp = torch.cat([block(b) for b in perms[l][0:8]])[:S]
            vp = torch.cat([block(b) for b in perms[l][::-1][0:8]])[:S]
            yield Write(kp, vp, lin_pos(-S, S), ring=l)
        for c in range(chunks):
            if c == 4:
                for l in range(layers):
                    yield Reset(4 * N, ring=l)
            start = (c if c < 4 else c - 4) * N
            pos = lin_pos(start, N)
            for l in range(layers):
                p = perms[l]
                yield Write(block(p[8 + 6 * c]), block(p[9 + 6 * c]), pos, ring=l)
                for ps in range(passes):
                    yield Attend(block(p[10 + 6 * c + ps]), pos, ring=l,
                                 tag=f"c{c}p{ps}")
    return Workload("chunk", shape, layers, ops(),
                    note="inputs drawn from a 64-block pool by per-ring permutations")


SWEEP_HEADS = (8, 24, 48)
SWEEP_DIMS = (64, 128)
SWEEP_SLOTS = (1447, 2894, 5788, 11576)
SWEEP_RESET = 42


def sweep_new_tokens(n_slots: int) -> int:
    return int(math.floor(n_slots * NEW_TOKENS / SLOTS + 0.5))


def sweep_grid(n: int):
    wg = int(math.ceil(math.sqrt(n * 1088 / 704)))
    hg = int(math.ceil(n / wg))
    return hg, wg


def sweep_positions(t: int, n: int) -> np.ndarray:
    hg, wg = sweep_grid(n)
    i = np.arange(n)
    return np.stack([np.full(n, t), i // wg, i % wg], axis=1).astype(np.int32)


def sweep(heads: int, head_dim: int, n_slots: int) -> Workload:
    """Frames t = 0 .. F-1 of N tokens fill the ring (F = ceil(S/N), so it
    wraps), then frame F is written, the ring is reset by 42 frames on the
    temporal axis and frame F's queries attend at t = F - 42."""
    N = sweep_new_tokens(n_slots)
    F = -(-n_slots // N)
    hg, wg = sweep_grid(N)
    dims = (head_dim // 4, 3 * head_dim // 8, 3 * head_dim // 8)
    shape = Shape(heads, head_dim, n_slots, dims, (-64, 0, 0), (128, hg, wg))

    def ops():
        g = rng(4, heads, head_dim, n_slots)
        for t in range(F):
            yield Write(normal_bf16(g, (N, heads, head_dim)),
                        normal_bf16(g, (N, heads, head_dim)), sweep_positions(t, N))
        k = normal_bf16(g, (N, heads, head_dim))
        v = normal_bf16(g, (N, heads, head_dim))
        q = normal_bf16(g, (N, heads, head_dim))
        yield Write(k, v, sweep_positions(F, N))
        yield Reset(SWEEP_RESET)
        yield Attend(q, sweep_positions(F - SWEEP_RESET, N), tag="sweep")
    return Workload(f"sweep_h{heads}_d{head_dim}_s{n_slots}", shape, 1, ops())


def sweep_shapes():
    return [(h, d, s) for h in SWEEP_HEADS for d in SWEEP_DIMS for s in SWEEP_SLOTS]


GLOBAL_SLOTS = 1246
WINDOW_FRAMES = 6
WINDOWED_PERIOD = 7
WINDOWED_STEPS = 10


def windowed(steps: int = WINDOWED_STEPS, period: int = WINDOWED_PERIOD) -> Workload:
    """1,246 global tokens at temporal positions -1246 .. -1, written once;
    then step s writes a 757-token frame at (s mod period)*757 + i and attends
    757 queries at those positions; before steps period, 2*period, ... the
    window is reset by period*757.  Seed 5; 1% of the channels x8."""
    H, D, G, N = 24, 128, GLOBAL_SLOTS, NEW_TOKENS
    S = G + WINDOW_FRAMES * N
    dshift = period * N
    shape = Shape(H, D, S, (D,), (-G,), (G + dshift,), n_global=G)

    def ops():
        g = rng(5)
        ch = outlier_channels(g, H, D)
        yield WriteGlobal(normal_bf16(g, (G, H, D), ch), normal_bf16(g, (G, H, D), ch), lin_pos(-G, G))
        for s in range(steps):
            if s > 0 and s % period == 0:
                yield Reset(dshift)
            pos = lin_pos((s % period) * N, N)
            k = normal_bf16(g, (N, H, D), ch)
            v = normal_bf16(g, (N, H, D), ch)
            q = normal_bf16(g, (N, H, D), ch)
            yield Write(k, v, pos)
            yield Attend(q, pos, tag=f"s{s}")
    return Workload("windowed", shape, 1, ops())


def windowed_tiny(steps: int = 8, period: int = 4) -> Workload:
    """H=2, D=64, 10 globals (t = -1, on a 4-wide grid), a window of three
    16-token frames (t = s mod period, a 4x4 grid); reset by period before
    step period; an attend after every write."""
    H, D, G, N = 2, 64, 10, 16
    S = G + 3 * N
    shape = Shape(H, D, S, (16, 24, 24), (-1, 0, 0), (period + 1, 4, 4), n_global=G)

    def grid(t, n):
        i = np.arange(n)
        return np.stack([np.full(n, t), i // 4, i % 4], axis=1).astype(np.int32)

    def ops():
        g = rng(6)
        yield WriteGlobal(normal_bf16(g, (G, H, D)), normal_bf16(g, (G, H, D)), grid(-1, G))
        for s in range(steps):
            if s > 0 and s % period == 0:
                yield Reset(period)
            pos = grid(s % period, N)
            yield Write(normal_bf16(g, (N, H, D)), normal_bf16(g, (N, H, D)), pos)
            yield Attend(normal_bf16(g, (N, H, D)), pos, tag=f"t{s}")
    return Workload("windowed_tiny", shape, 1, ops())


STATIC_MARGIN = 1.5
CALIBRATION_STEPS = 6


def _static(wl: Workload, big_step=None) -> Workload:
    """``wl`` on a ring with per-head fixed scales: calibrate after the
    sixth window write; the K and V of write ``big_step`` (if any) scaled x3."""
    shape = Shape(**{**wl.shape.__dict__, "scale_mode": "static"})

    def ops():
        n_writes = 0
        for op in wl.ops:
            if isinstance(op, Write):
                if n_writes == CALIBRATION_STEPS:
                    yield Calibrate(STATIC_MARGIN)
                if n_writes == big_step:
                    op = Write(op.k * 3, op.v * 3, op.pos, op.ring)   # rounded to bf16; both sides read it
                n_writes += 1
            yield op
    return Workload("static_" + wl.name, shape, wl.n_rings, ops())


def static_scales(steps: int = WINDOWED_STEPS) -> Workload:
    """The paper's layout and input recipe with the paper's scales."""
    return _static(windowed(steps))


def static_scales_tiny() -> Workload:
    """windowed_tiny over ten steps, reset by 7 before step 7 (after the calibration)."""
    return _static(windowed_tiny(steps=10, period=7), big_step=8)
