"""GPU parity of the three kernels against the oracle, through the C ABI.

Every workload of ``synth`` is replayed call by call on the library and on the
oracle (tests/replay.py): ring state, codes and scales bit for bit after every
write and reset; attention outputs within max-abs 1e-2 and mean-abs 1e-3 of the
fp64 oracle over its own FP8 cache.
"""
import numpy as np
import pytest
import torch

import synth
from replay import replay

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_ring_kv_gb300 import kvring
    kvring.load()


def test_tiny_ring_wraps_and_resets():
    rep = replay(synth.tiny())
    assert rep.writes == 6 and rep.resets == 1 and rep.attend_checked == 6
    print("tiny", rep)


def test_tiny_ring_bf16_output():
    rep = replay(synth.tiny(), out_f32=False)
    assert rep.attend_checked == 6


def test_single_call_at_paper_shape():
    rep = replay(synth.single())
    assert rep.attend_checked == 1
    print("single", rep.attend_stats, f"{rep.seconds:.1f}s")


def test_sustained_with_resets():
    keep = {"s0", "s1", "s41", "s42", "s43", "s83", "after_reset"}
    rep = replay(synth.sustained(), cache_every=7, attend_filter=lambda t: t in keep)
    assert rep.resets == 2 and rep.attend_checked == len(keep)
    print("sustained", rep.attend_stats, f"{rep.seconds:.1f}s")


def test_chunk_workload_sampled_rings():
    keep = {f"c{c}p{p}" for c in (0, 3, 4, 7) for p in (0, 3)}
    rep = replay(synth.chunk(), cache_every=0, oracle_rings=(0, 59), attend_filter=lambda t: t in keep,
                 attend_heads=(0, 11, 23))
    assert rep.attends == 60 * 8 * 4 and rep.attend_checked == 2 * len(keep)
    print("chunk", rep.worst_max_abs, rep.worst_mean_abs, f"{rep.seconds:.1f}s")


@pytest.mark.parametrize("heads,head_dim,n_slots", synth.sweep_shapes())
def test_sweep(heads, head_dim, n_slots):
    rep = replay(synth.sweep(heads, head_dim, n_slots), cache_every=3)
    assert rep.attend_checked == 1


@pytest.mark.parametrize("heads,head_dim", [(64, 128), (128, 64)])
def test_largest_head_counts(heads, head_dim):
    """The largest head counts the library accepts (2 * heads * head_dim / 16 =
    1024: one 512-thread block per token in the write and query kernels),
    through the sweep workload on a 1,447-slot ring that wraps: every cache
    bit for bit, the attention of all heads within the tolerance."""
    rep = replay(synth.sweep(heads, head_dim, 1447), cache_every=1)
    assert rep.writes == 9 and rep.resets == 1 and rep.attend_checked == 1


def _tile_exact():
    """A 1,024-slot ring (eight 128-slot key tiles) whose valid count is a
    whole number of tiles at every attend (896, then 1,024, then full after
    wrapping writes), queried by exactly one and two 128-query tiles: the
    kernels' paths with no partial key or query tile.  Seed 12."""
    H, D, S = 8, 128, 1024
    shape = synth.Shape(H, D, S, (D,), (0,), (4096,))

    def ops():
        g = synth.rng(12)
        yield synth.Write(synth.normal_bf16(g, (896, H, D)), synth.normal_bf16(g, (896, H, D)), synth.lin_pos(0, 896))
        yield synth.Attend(synth.normal_bf16(g, (128, H, D)), synth.lin_pos(768, 128), tag="n896_q128")
        for t, n_q in ((0, 128), (1, 256)):
            start = 896 + 128 * t
            yield synth.Write(synth.normal_bf16(g, (128, H, D)), synth.normal_bf16(g, (128, H, D)),
                              synth.lin_pos(start, 128))
            yield synth.Attend(synth.normal_bf16(g, (n_q, H, D)), synth.lin_pos(start + 128 - n_q, n_q),
                               tag=f"w{t}_q{n_q}")
        yield synth.Reset(512)
        yield synth.Attend(synth.normal_bf16(g, (256, H, D)), synth.lin_pos(400, 256), tag="after_reset")
    return synth.Workload("tile_exact", shape, 1, ops())


def test_whole_tiles_of_slots_and_queries():
    rep = replay(_tile_exact(), cache_every=1)
    assert rep.writes == 3 and rep.resets == 1 and rep.attend_checked == 4


def test_global_slots_tiny_3axis():
    """Global slots written once, a 3-frame window ring that wraps twice, a
    reset that must leave the globals alone; everything compared after every
    call."""
    rep = replay(synth.windowed_tiny())
    assert rep.writes == 9 and rep.resets == 1 and rep.attend_checked == 8
    print("windowed_tiny", rep.attend_stats)


def test_global_slots_tiny_bf16_output():
    rep = replay(synth.windowed_tiny(), out_f32=False)
    assert rep.attend_checked == 8


def test_global_slots_at_paper_layout():
    """1,246 globals + six 757-token frames (5,788 slots), ten steps with a
    reset before step 7: cache bit for bit after every call; attention
    checked when the window is first full, after the first wrap, right after
    the reset and at the end."""
    keep = {"s0", "s5", "s6", "s7", "s9"}
    rep = replay(synth.windowed(), attend_filter=lambda t: t in keep)
    assert rep.writes == 11 and rep.resets == 1 and rep.attend_checked == len(keep)
    print("windowed", rep.attend_stats, f"{rep.seconds:.1f}s")


def test_static_scales_tiny():
    """Per-head scales fixed by a calibration on entering the seventh step,
    a reset after it (clamping), a step whose values pass the range; every
    call compared."""
    rep = replay(synth.static_scales_tiny())
    assert rep.resets == 1 and rep.attend_checked == 10
    print("static_tiny", rep.attend_stats)


def test_static_scales_at_paper_layout():
    keep = {"s5", "s6", "s7", "s8", "s9"}
    rep = replay(synth.static_scales(), attend_filter=lambda t: t in keep)
    assert rep.resets == 1 and rep.attend_checked == len(keep)
    print("static", rep.attend_stats, f"{rep.seconds:.1f}s")
