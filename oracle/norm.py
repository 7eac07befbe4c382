"""RMS normalisation of Q and K ahead of RoPE, as fixed rounding steps.

Runway Characters paper, §4.4 "Fused pre-attention" and Appendix G: each
block RMS-normalises the new tokens' Q and K before RoPE and the FP8 write;
the fused kernels square in fp32.  Where the paper leaves a step open this
module takes one plain reading, each step one rounding:

* the norm runs over each head's D channels (heads are split across
  tensor-parallel ranks, and the paper's block needs only the one all-reduce
  after its output projection);
* S = sum_d x_d^2, exact, rounded once to fp32 (so no summation order can
  change it);  ms = fl32(S / D);  v = fl32(ms + eps);
* rstd = 1 / sqrt(v) rounded once to fp32 (correctly rounded);
* y_d = bf16(fl32(fl32(x_d * rstd) * gamma_d)), rounded to nearest even:
  the normalised values leave the fused step as bf16, the precision in which
  the paper compares them with the unfused reference.

Rounding a rational once to fp32 is done here in exact integer arithmetic
(``rn32``); a sum of floats is taken exactly with ``math.fsum`` (correctly
rounded to fp64) and re-rounded to fp32 only where that cannot round twice.
"""
import math
from fractions import Fraction

import numpy as np


def rn32(q: Fraction) -> np.float32:
    """The float32 nearest to the rational ``q`` (ties to even); normal
    range only (|q| in [2^-126, 2^128)) or zero."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()      # 2^(e-1) < q < 2^(e+1)
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    # q = m * 2^(e-23) with m in [2^23, 2^24)
    scaled = q / Fraction(2) ** (e - 23)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    if not -126 <= e + (1 if m == 2 ** 24 else 0) <= 127:
        raise ValueError("outside the normal float32 range")
    return np.float32(sign * math.ldexp(m, e - 23))


def _is_fp32_midpoint(x: float) -> bool:
    """True if the fp64 value x lies exactly halfway between two adjacent
    fp32 values (normal range)."""
    if x == 0 or not math.isfinite(x):
        return False
    m, e = math.frexp(abs(x))                      # x = m 2^e, m in [0.5, 1)
    k = m * 2.0 ** 25                              # 25 significant bits: the midpoint grid
    return k == int(k) and int(k) % 2 == 1


def sum_sq_f32(row) -> np.float32:
    """fl32 of the exact sum of squares of a row of float32 values."""
    vals = [float(t) * float(t) for t in np.asarray(row, np.float32)]   # exact in fp64 (48-bit products)
    s = math.fsum(vals)                                                  # the exact sum, rounded to fp64
    if _is_fp32_midpoint(s):                                             # fp64 rounding may have moved a tie
        return rn32(sum(Fraction(v) for v in vals))
    return np.float32(s)


def rsqrt_rn32(v, start=None) -> np.float32:
    """fl32 of 1/sqrt(v), correctly rounded, for a float32 v > 0.  The fp64
    estimate (or ``start``) is moved to the nearest fp32 by exact tests."""
    v = np.float32(v)
    if not v > 0:
        raise ValueError("rsqrt of a non-positive value")
    r = np.float32(1.0 / math.sqrt(float(v))) if start is None else np.float32(start)
    fv = Fraction(float(v))
    # r is the nearest fp32 to 1/sqrt(v) iff 1/sqrt(v) lies between the
    # midpoints to r's neighbours; y^2 v grows with y > 0, so for a midpoint
    # m: 1/sqrt(v) < m  <=>  m^2 v > 1 (no midpoint is hit exactly: it would
    # make v = 1/m^2 a non-dyadic number)
    for _ in range(4):
        lo = Fraction(float(np.nextafter(r, np.float32(0.0)))) / 2 + Fraction(float(r)) / 2
        hi = Fraction(float(r)) / 2 + Fraction(float(np.nextafter(r, np.float32(np.inf)))) / 2
        if lo * lo * fv > 1:           # 1/sqrt(v) < lo: step down
            r = np.nextafter(r, np.float32(0.0))
        elif hi * hi * fv < 1:         # 1/sqrt(v) > hi: step up
            r = np.nextafter(r, np.float32(np.inf))
        else:
            return np.float32(r)
    raise AssertionError("rsqrt_rn32 did not settle")


def round_bf16(x) -> np.ndarray:
    """float32 -> nearest bfloat16 value (ties to even), as float32."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def rms_norm_bf16(x, gamma, eps=1e-6) -> np.ndarray:
    """x: float32 [..., D] (bf16 values); gamma: float32 broadcastable to x
    (bf16 values); returns the normalised rows as float32 holding bf16 values."""
    x = np.asarray(x, np.float32)
    gamma = np.broadcast_to(np.asarray(gamma, np.float32), x.shape)
    D = x.shape[-1]
    eps32 = np.float32(eps)
    flat = x.reshape(-1, D)
    rstd = np.empty(flat.shape[0], np.float32)
    for i, row in enumerate(flat):
        ms = np.float32(sum_sq_f32(row) / np.float32(D))
        rstd[i] = rsqrt_rn32(np.float32(ms + eps32))
    t = (x * rstd.reshape(x.shape[:-1])[..., None]).astype(np.float32)
    return round_bf16((t * gamma).astype(np.float32))
