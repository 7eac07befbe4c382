"""OCP E4M3 ("FN") codec, written from the bit definition of the format.

The paper stores K and V as float8_e4m3 (Runway Characters paper, §4.3 "FP8 at
write") and clamps/saturates out-of-range values to the FP8 range (§4.2 and
Appendix G "Cache update and position reset").  The format is the OCP 8-bit
E4M3 variant without infinities: 1 sign bit, 4 exponent bits (bias 7), 3
mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; the single pattern
S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448.

Encoding is round-to-nearest, ties to the even code (mantissa LSB 0), with
saturation: any finite or infinite input whose magnitude rounds above 448 is
clamped to +-448.  The sign of the input is kept (a negative input that rounds
to zero gives -0, code 0x80).  NaN encodes as 0x7F with the input's sign.
"""
import numpy as np

E4M3_MAX = 448.0
N_FINITE_POS = 127          # codes 0x00..0x7E are the finite non-negative values


def _decode_one(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:                       # subnormal: (m/8) * 2^(1-bias)
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


#: value of each of the 256 codes, float64 (exact: every value is a short dyadic)
E4M3_VALUES = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)

# the finite non-negative values in code order; they increase with the code
_POS = E4M3_VALUES[:N_FINITE_POS].copy()
assert np.all(np.diff(_POS) > 0)


def decode(codes) -> np.ndarray:
    """Codes (uint8 array) -> float64 values."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def encode_rn_satfinite(x) -> np.ndarray:
    """float32 (or float64 holding float32 values) -> uint8 e4m3 codes.

    Round to nearest, ties to even, saturate to +-448, keep the sign of zero.
    """
    x = np.asarray(x)
    xf = x.astype(np.float64)
    neg = np.signbit(xf)
    mag = np.abs(xf)
    nan = np.isnan(mag)
    mag = np.where(nan, 0.0, mag)
    sat = mag >= E4M3_MAX                      # includes +inf
    m = np.where(sat, 0.0, mag)
    # index of the first table value >= m; the candidates are that one and the one below
    hi = np.searchsorted(_POS, m, side="left")
    hi = np.minimum(hi, N_FINITE_POS - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS[hi] - m                       # exact in float64
    d_lo = m - _POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(m == _POS[hi], hi, code)   # exact hits
    code = np.where(sat, N_FINITE_POS - 1, code)
    code = np.where(nan, 0x7F, code)
    code = code.astype(np.uint8) | (neg.astype(np.uint8) << 7)
    return code.astype(np.uint8)


def spacing(codes) -> np.ndarray:
    """Distance from |value(code)| to the next larger finite magnitude (float64).

    For 448 (the top code) the spacing below it (32) is returned.
    """
    c = (np.asarray(codes, dtype=np.uint8) & 0x7F).astype(np.int64)
    c = np.minimum(c, N_FINITE_POS - 1)
    up = np.minimum(c + 1, N_FINITE_POS - 1)
    gap = _POS[up] - _POS[c]
    return np.where(c == N_FINITE_POS - 1, _POS[c] - _POS[np.maximum(c - 1, 0)], gap)


def ordinal(codes) -> np.ndarray:
    """Signed ordinal of each finite code: consecutive values differ by 1 and
    +0 / -0 both map to 0, so ``|ordinal(a) - ordinal(b)|`` counts e4m3 ulps."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def ulp_distance(a, b) -> np.ndarray:
    return np.abs(ordinal(a) - ordinal(b))
