"""Per-token-per-head absmax quantisation to e4m3.

The paper quantises K and V to float8_e4m3 once, at write time (Runway
Characters paper, §4.3 "FP8 at write"; Appendix G), and quantises the queries
once per call (§4.3: only the queries are quantized per call).  The scale
granularity used here is one fp32 scale per (token, head) row, set from that
row's absolute maximum so the row uses the whole e4m3 range up to 448.

The decision that yields an integer code is taken in fp32, the precision the
paper gives for the cached-key arithmetic (§4.2: keys are rotated in fp32):

    amax  = max_i |x_i|                     (exact)
    scale = fl32(amax / 448)                (IEEE fp32 division)
    inv   = fl32(448 / amax)                (IEEE fp32 division)
    code_i = e4m3_rn_satfinite(fl32(x_i * inv))

A row whose amax is 0 gets scale 0 and all codes +0.  Dequantisation is
code * scale, in fp32 (``dequantize_rows``) or exactly in fp64
(``dequantize_rows_f64``).
"""
import numpy as np

from . import e4m3

F32_448 = np.float32(448.0)


def quantize_rows(x):
    """x: float32 [..., D] -> (codes uint8 [..., D], scale float32 [...])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    zero = amax == 0
    safe = np.where(zero, np.float32(1.0), amax).astype(np.float32)
    scale = (safe / F32_448).astype(np.float32)
    inv = (F32_448 / safe).astype(np.float32)
    y = (x * inv[..., None]).astype(np.float32)
    codes = e4m3.encode_rn_satfinite(y)
    codes = np.where(zero[..., None], np.uint8(0), codes).astype(np.uint8)
    scale = np.where(zero, np.float32(0.0), scale).astype(np.float32)
    return codes, scale


def dequantize_rows(codes, scale):
    """fp32 dequantisation: fl32(value(code) * scale)."""
    v = e4m3.decode(codes).astype(np.float32)
    return (v * np.asarray(scale, dtype=np.float32)[..., None]).astype(np.float32)


def dequantize_rows_f64(codes, scale):
    """Exact dequantisation in fp64 (the product of an e4m3 value and an fp32
    scale is exact in fp64)."""
    return e4m3.decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]


# --- per-head scales fixed once per session ------------------------------------
# The paper's own scheme (§4.3 "FP8 at write"; Appendix G): one scale per
# (cache, head) for K and one for V, set once per session from the absolute
# maximum of what the first steps wrote, times a margin of 1.5; later values
# beyond the range saturate, and a position reset keeps the scale and clamps.
#
#     a     = fl32(margin * amax)
#     scale = fl32(a / 448),  inv = fl32(448 / a)       (0 and 0 when a = 0)
#     code_i = e4m3_rn_satfinite(fl32(x_i * inv))       (+0 when inv = 0)

def static_scale(amax, margin=1.5):
    """Per-head amax (float32 [...]) -> (scale, inv), float32 [...]."""
    amax = np.asarray(amax, dtype=np.float32)
    a = (np.float32(margin) * amax).astype(np.float32)
    zero = a == 0
    safe = np.where(zero, np.float32(1.0), a).astype(np.float32)
    scale = np.where(zero, np.float32(0.0), (safe / F32_448).astype(np.float32)).astype(np.float32)
    inv = np.where(zero, np.float32(0.0), (F32_448 / safe).astype(np.float32)).astype(np.float32)
    return scale, inv


def quantize_rows_fixed(x, inv):
    """x: float32 [..., D]; inv: float32 [...] (one per row, broadcast) ->
    codes uint8 [..., D], saturating at +-448."""
    x = np.asarray(x, dtype=np.float32)
    inv = np.asarray(inv, dtype=np.float32)
    y = (x * inv[..., None]).astype(np.float32)
    codes = e4m3.encode_rn_satfinite(y)
    return np.where((inv == 0)[..., None], np.uint8(0), codes).astype(np.uint8)
