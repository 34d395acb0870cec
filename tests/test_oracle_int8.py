"""Pins of the oracle's INT8 key codec (``oracle/int8.py``): the integer grid
is reproduced exactly, midpoints round to the even integer, values beyond the
symmetric range clamp to +-127 and never to -128, the scale rule follows the
absmax reading, and the dequantised error stays within half a step."""

import numpy as np

from oracle import int8 as OI


def test_integer_grid_is_a_fixed_point():
    # every code value, given as an exact float, encodes to itself
    vals = np.arange(-127, 128, dtype=np.float32)
    assert np.array_equal(OI.int8_encode(vals).astype(np.int64), np.arange(-127, 128))


def test_midpoints_round_to_even():
    mids = np.arange(-126.5, 127.0, 1.0, dtype=np.float32)  # -126.5 .. 126.5
    got = OI.int8_encode(mids).astype(np.int64)
    lo = np.floor(mids).astype(np.int64)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want)
    # just off the midpoint goes to the nearer integer, whatever its parity
    assert OI.int8_encode(np.float32([2.5000002, 2.4999998, -3.5000002])).tolist() == [3, 2, -4]


def test_clamp_is_symmetric():
    got = OI.int8_encode(np.float32([127.4, 127.5, 128.0, 1e9, -127.5, -128.0, -1e9])).astype(np.int64)
    assert got.tolist() == [127, 127, 127, 127, -127, -127, -127]


def test_scale_rule_and_zero_block():
    x = np.float32([[0.5, -2.0], [1.25, 0.0]])
    codes, s = OI.quantize_block(x)
    assert s == np.float32(np.float32(2.0) / np.float32(127.0))
    # the absmax element maps to +-127 exactly
    assert codes[0, 1] == -127
    z_codes, z_s = OI.quantize_block(np.zeros((3, 4), np.float32))
    assert z_s == 1.0 and not z_codes.any()


def test_dequantisation_error_within_half_a_step():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 128)) * np.where(rng.random((64, 128)) < 0.01, 8.0, 1.0)).astype(np.float32)
    codes, s = OI.quantize_block(x)
    err = np.abs(OI.dequantize_block(codes, s) - x.astype(np.float64))
    # half a quantisation step, plus the rounding of the fp32 division
    assert err.max() <= 0.5 * float(s) * (1 + 1e-6) + 1e-12
    assert codes.min() >= -127 and codes.max() <= 127


def test_chunk_layout_matches_blocks():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 5, 3, 8)).astype(np.float32)  # [B, Lc, H, D]
    codes, scales = OI.quantize_chunk_bhld(x)
    assert codes.shape == (2, 3, 5, 8) and scales.shape == (2, 3)
    c12, s12 = OI.quantize_block(x[1, :, 2, :])
    assert np.array_equal(codes[1, 2], c12) and scales[1, 2] == s12
