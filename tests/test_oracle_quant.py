"""Pins of the oracle's per-token-per-head absmax quantisation."""
import numpy as np

from oracle import e4m3, quant


def test_row_max_maps_to_448():
    g = np.random.default_rng(0)
    x = (g.standard_normal((500, 4, 64)) * np.exp2(g.uniform(-20, 20, (500, 4, 1)))).astype(np.float32)
    codes, scale = quant.quantize_rows(x)
    idx = np.argmax(np.abs(x), axis=-1)
    top = np.take_along_axis(codes, idx[..., None], -1)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    # the top code carries the sign of the row's largest-magnitude element
    sgn = np.take_along_axis(x, idx[..., None], -1)[..., 0] < 0
    assert np.array_equal((top >> 7).astype(bool), sgn)
    # scale is amax/448 correctly rounded: fp64 division then one rounding gives the same
    amax = np.max(np.abs(x), -1)
    assert np.array_equal(scale, (amax.astype(np.float64) / 448.0).astype(np.float32))


def test_zero_row():
    x = np.zeros((3, 2, 16), np.float32)
    x[1, 0, 3] = -2.5
    codes, scale = quant.quantize_rows(x)
    assert scale[0, 0] == 0 and scale[2, 1] == 0 and np.all(codes[0] == 0)
    assert scale[1, 0] == np.float32(2.5 / 448)
    assert codes[1, 0, 3] == 0xFE


def test_power_of_two_amax_is_a_plain_cast():
    # amax = 448 -> scale 1, inv 1: the codes are the plain cast of x
    g = np.random.default_rng(1)
    x = g.uniform(-448, 448, (64, 32)).astype(np.float32)
    x[:, 0] = 448.0
    codes, scale = quant.quantize_rows(x)
    assert np.all(scale == 1.0)
    assert np.array_equal(codes, e4m3.encode_rn_satfinite(x))


def test_error_bound():
    # |dequant - x| <= half a code spacing (in the scaled domain) per element
    g = np.random.default_rng(2)
    x = (g.standard_normal((2000, 128)) * g.choice([1, 8], (1, 128), p=[0.99, 0.01])).astype(np.float32)
    codes, scale = quant.quantize_rows(x)
    deq = quant.dequantize_rows_f64(codes, scale)
    inv = (np.float32(448) / np.max(np.abs(x), -1)).astype(np.float32)
    y = (x * inv[:, None]).astype(np.float64)                      # scaled value that was rounded
    vals = e4m3.decode(codes)
    # neighbour spacing on either side of the chosen code
    c = codes & 0x7F
    lo_gap = np.where(c > 0, e4m3.E4M3_VALUES[c] - e4m3.E4M3_VALUES[np.maximum(c.astype(int) - 1, 0)], 2.0 ** -9)
    hi_gap = e4m3.spacing(codes)
    assert np.all(np.abs(np.abs(y) - np.abs(vals)) <= np.maximum(lo_gap, hi_gap) / 2 + 1e-12)
    # and in the original units the relative error of normal-range values is <= 2^-4
    normal = np.abs(vals) >= 2.0 ** -6
    rel = np.abs(deq - x) / np.abs(x)
    assert np.all(rel[normal] <= 2.0 ** -4 * (1 + 1e-6))


def test_dequant_f32_is_one_rounding_of_exact():
    g = np.random.default_rng(3)
    codes = g.integers(0, 256, (100, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10
    scale = np.exp2(g.uniform(-10, 3, 100)).astype(np.float32)
    assert np.array_equal(quant.dequantize_rows(codes, scale),
                          quant.dequantize_rows_f64(codes, scale).astype(np.float32))
