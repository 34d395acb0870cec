"""E4M3 codec and per-(head, chunk) absmax quantiser -- oracle (test infrastructure).

Not for the product path; see the package docstring.

Sources
-------
* The E4M3 format itself follows the OCP "OFP8 Formats for Deep Learning"
  specification: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
  subnormals at exponent field 0, no infinities, and the single NaN pattern
  S.1111.111 per sign, so the largest finite magnitude is S.1111.110 = 448.
* The use of an 8-bit KV cache comes from "Matrix-Game 4.0: Harnessing Video
  Models for Real-Time Playable Game Worlds", section "技术新颖性" (keys and
  values of each KV-window interval are cached in 8 bits, and only the changed
  interval is re-quantised) and section "前置知识 / FP8 量化与 CUDA Graph".
  The pages do not fix the scale rule; the reading used here is one fp32
  absmax scale per (batch, head, chunk) and per tensor (K or V):
  ``scale = amax / 448`` (fp32, round-to-nearest-even division; ``scale = 1``
  when ``amax == 0``), ``code = E4M3_RNE_satfinite(x / scale)`` with the
  division again in fp32, and ``x_hat = value(code) * scale``.

Conversion from fp32 rounds to nearest with ties to the even code, saturates
finite values above 448 in magnitude to +-448 ("satfinite"), keeps the sign of
values that round to zero, and maps NaN to the NaN pattern.
"""

from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def e4m3_decode_code(code: int) -> float:
    """Value of one E4M3 code (0..255) from its bit fields, as a Python float."""
    code = int(code) & 0xFF
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return math.nan
    if exp_field == 0:
        # subnormal: 0.mmm * 2^(1 - bias)
        return sign * (mant / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


# Table of the 127 non-negative finite magnitudes, indexed by code 0..126.
# Codes 0..126 are strictly increasing in value (sign-magnitude encoding).
_POS_VALUES = np.array([e4m3_decode_code(c) for c in range(127)], dtype=np.float64)
_DECODE_TABLE = np.array([e4m3_decode_code(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Vectorised decode of uint8 codes to float64 values."""
    return _DECODE_TABLE[np.asarray(codes, dtype=np.uint8).astype(np.int64)]


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round float32 values to E4M3 codes: nearest, ties to even, satfinite.

    ``x`` is first taken as float32 (its exact value is what is rounded).
    Returns uint8 codes with the same shape.
    """
    x32 = np.asarray(x, dtype=np.float32)
    a = np.abs(x32).astype(np.float64)  # exact
    neg = np.signbit(x32)
    nan = np.isnan(x32)
    a = np.where(nan, 0.0, a)
    # Nearest representable magnitude.  hi = first table index with value >= a.
    hi = np.searchsorted(_POS_VALUES, a, side="left")
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    v_hi = _POS_VALUES[hi]
    v_lo = _POS_VALUES[lo]
    d_hi = v_hi - a  # exact in fp64: both operands have short mantissas
    d_lo = a - v_lo
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(a >= v_hi, hi, np.where(pick_hi, hi, lo))
    # satfinite: anything above the largest finite magnitude becomes 448 (code 126)
    mag = np.where(a > E4M3_MAX, 126, mag).astype(np.int64)
    code = mag | np.where(neg, 0x80, 0)
    code = np.where(nan, E4M3_NAN_CODE, code)
    return code.astype(np.uint8)


def absmax_scale(x: np.ndarray) -> np.float32:
    """fp32 scale of one (batch, head, chunk) block: amax / 448, or 1 if amax is 0."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / np.float32(E4M3_MAX))  # fp32 / fp32 -> fp32, IEEE RN


def quantize_block(x: np.ndarray) -> tuple[np.ndarray, np.float32]:
    """Quantise one block (e.g. one chunk of one head, shape [Lc, D]).

    Returns (codes uint8 with x's shape, fp32 scale).
    """
    x32 = np.asarray(x, dtype=np.float32)
    s = absmax_scale(x32)
    codes = e4m3_encode((x32 / s).astype(np.float32))  # fp32 division, IEEE RN
    return codes, s


def dequantize_block(codes: np.ndarray, scale: float) -> np.ndarray:
    """x_hat = value(code) * scale, in float64 (exact product)."""
    return e4m3_decode(codes) * np.float64(np.float32(scale))


def quantize_chunk_bhld(x_blhd: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantise a token-major chunk ``[B, Lc, H, D]`` per (batch, head).

    Returns codes ``[B, H, Lc, D]`` (head-major, like a ring slot) and scales
    ``[B, H]`` (fp32).
    """
    x = np.asarray(x_blhd, dtype=np.float32)
    B, Lc, H, D = x.shape
    codes = np.empty((B, H, Lc, D), dtype=np.uint8)
    scales = np.empty((B, H), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            c, s = quantize_block(x[b, :, h, :])
            codes[b, h] = c
            scales[b, h] = s
    return codes, scales
