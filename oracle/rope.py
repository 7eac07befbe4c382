"""Rotary position embedding (RoPE), its fp32 tables and the delta rotation.

Runway Characters paper, §4.2 "RoPE at write, and a delta rotation at reset"
and Appendix G: RoPE is applied once to each new token's Q and K before the
cache write; the angle of frequency j for temporal index t is
theta_j(t) = omega_j * (a*t + b) (here a = 1, b = 0, positions are integers);
at a reset every cached key is rotated by omega_j * a * Delta on the temporal
frequencies only, in fp32, and re-quantised.  RoPE itself is the rotary
embedding of Su et al. (RoFormer), cited by the paper.

Layout (one reading of the paper, which does not fix it): head_dim D is split
into ``n_axes`` consecutive axis blocks of widths ``axis_dims`` (axis 0 =
temporal); inside axis a (offset o_a, width d_a) pair j occupies channels
(o_a + 2j, o_a + 2j + 1) and rotates by theta = pos_a * omega_{a,j} with
omega_{a,j} = base^(-2j/d_a).  A pair (x0, x1) maps to
(x0 cos(theta) - x1 sin(theta), x0 sin(theta) + x1 cos(theta)).

Two versions:

* ``rope_f64`` -- the definition in fp64 (for the mathematical pins).
* ``rope_f32`` -- the rotation in fp32 arithmetic (the paper's precision for
  cached keys): cos and sin are the fp64 values of the exact angle rounded to
  fp32 once, and every product and sum is one IEEE fp32 operation:
  x0' = fl32(fl32(x0*c) - fl32(x1*s)),  x1' = fl32(fl32(x0*s) + fl32(x1*c)).
"""
import numpy as np


def frequencies(d_axis: int, base: float) -> np.ndarray:
    """omega_j = base^(-2j/d_axis), j = 0 .. d_axis/2 - 1 (fp64)."""
    j = np.arange(d_axis // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * j / d_axis)


def axis_offsets(axis_dims):
    off, o = [], 0
    for d in axis_dims:
        off.append(o)
        o += d
    return off


def cos_sin_f32(pos, omega):
    """fl32(cos(pos*omega)), fl32(sin(pos*omega)) with the angle formed in fp64.

    pos: int array [...]; omega: float64 [J] -> two float32 arrays [..., J]."""
    theta = np.asarray(pos, dtype=np.float64)[..., None] * omega
    return np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)


def rope_table_f32(d_axis, base, pos_min, pos_count):
    """fp32 cos/sin for positions pos_min .. pos_min+pos_count-1 of one axis:
    float32 [pos_count, d_axis/2, 2] holding (cos, sin)."""
    pos = np.arange(pos_min, pos_min + pos_count, dtype=np.int64)
    c, s = cos_sin_f32(pos, frequencies(d_axis, base))
    return np.stack([c, s], axis=-1)


def _rotate_pairs_f32(x, c, s):
    """x float32 [..., 2J] interleaved pairs; c, s float32 broadcastable [..., J]."""
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    y0 = (x0 * c).astype(np.float32) - (x1 * s).astype(np.float32)
    y1 = (x0 * s).astype(np.float32) + (x1 * c).astype(np.float32)
    out = np.empty_like(x)
    out[..., 0::2] = y0.astype(np.float32)
    out[..., 1::2] = y1.astype(np.float32)
    return out


def rope_f32(x, pos, axis_dims, base):
    """RoPE in fp32.  x: float32 [N, H, D]; pos: int [N, n_axes]."""
    x = np.asarray(x, dtype=np.float32)
    pos = np.asarray(pos).reshape(x.shape[0], len(axis_dims))
    out = x.copy()
    for a, (o, d) in enumerate(zip(axis_offsets(axis_dims), axis_dims)):
        c, s = cos_sin_f32(pos[:, a], frequencies(d, base))      # [N, d/2]
        out[..., o:o + d] = _rotate_pairs_f32(x[..., o:o + d], c[:, None, :], s[:, None, :])
    return out


def rope_f64(x, pos, axis_dims, base):
    """RoPE in fp64.  x: [N, H, D]; pos: int [N, n_axes]."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.asarray(pos).reshape(x.shape[0], len(axis_dims))
    out = x.copy()
    for a, (o, d) in enumerate(zip(axis_offsets(axis_dims), axis_dims)):
        theta = pos[:, a].astype(np.float64)[:, None] * frequencies(d, base)
        c = np.cos(theta)[:, None, :]
        s = np.sin(theta)[:, None, :]
        x0 = x[..., o:o + d:2]
        x1 = x[..., o + 1:o + d:2]
        out[..., o:o + d:2] = x0 * c - x1 * s
        out[..., o + 1:o + d:2] = x0 * s + x1 * c
    return out


def delta_cos_sin_f32(d, d_temporal, base):
    """The reset rotation R(-d) of the temporal axis: fp32 (cos, sin) of the
    angle -d * omega_{0,j}, formed in fp64 and rounded once.  float32 [d_t/2] x2."""
    return cos_sin_f32(np.int64(-d), frequencies(d_temporal, base))


def rotate_temporal_f32(x, c, s, d_temporal):
    """Rotate the temporal pairs (channels 0 .. d_temporal-1) of x [..., D] in
    fp32 by the angles whose fp32 cosines/sines are c, s; other channels are
    left as they are."""
    x = np.asarray(x, dtype=np.float32)
    out = x.copy()
    out[..., :d_temporal] = _rotate_pairs_f32(x[..., :d_temporal], c, s)
    return out


def rotate_temporal_f64(x, d, d_temporal, base):
    """R(-d) on the temporal pairs in fp64."""
    x = np.asarray(x, dtype=np.float64)
    theta = -np.float64(d) * frequencies(d_temporal, base)
    c, s = np.cos(theta), np.sin(theta)
    out = x.copy()
    x0 = x[..., 0:d_temporal:2]
    x1 = x[..., 1:d_temporal:2]
    out[..., 0:d_temporal:2] = x0 * c - x1 * s
    out[..., 1:d_temporal:2] = x0 * s + x1 * c
    return out
