"""Symmetric INT8 codec and per-(head, chunk) absmax quantiser for cached keys
-- oracle (test infrastructure).

Not for the product path; see the package docstring.

Source: "Matrix-Game 4.0: Harnessing Video Models for Real-Time Playable Game
Worlds", section "技术新颖性": every KV-window interval caches its keys in
INT8 and its values in FP8, and only the interval that changed is
re-quantised.  The pages fix neither the integer range nor the scale rule;
the reading used here mirrors the FP8 reading (one fp32 scale per batch,
head and chunk):

* ``scale = amax / 127`` (fp32, IEEE round-to-nearest division; ``scale = 1``
  when ``amax == 0``), so the code range is symmetric and -128 is unused;
* ``code = clamp(round_half_even(x / scale), -127, 127)`` with the division
  in fp32 (|x| <= amax keeps x / scale within [-127, 127] up to rounding of
  the division; the clamp only absorbs that rounding);
* ``x_hat = code * scale``.

Values are cached as an INT8 byte (two's complement) in the ring's byte
storage; the values of the same chunk use the E4M3 codec of ``oracle.fp8``.
"""

from __future__ import annotations

import numpy as np

INT8_MAX = 127.0


def int8_scale(x: np.ndarray) -> np.float32:
    """fp32 scale of one block: amax / 127, or 1 if amax is 0."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / np.float32(INT8_MAX))  # fp32 / fp32 -> fp32, IEEE RN


def int8_encode(y: np.ndarray) -> np.ndarray:
    """Round already-scaled float32 values to int8 codes: nearest, ties to even,
    clamped to [-127, 127]."""
    y64 = np.asarray(y, dtype=np.float32).astype(np.float64)  # exact
    r = np.rint(y64)  # numpy rint: round half to even
    return np.clip(r, -INT8_MAX, INT8_MAX).astype(np.int8)


def quantize_block(x: np.ndarray) -> tuple[np.ndarray, np.float32]:
    """Quantise one block (one chunk of one head, shape [Lc, D]).

    Returns (int8 codes with x's shape, fp32 scale)."""
    x32 = np.asarray(x, dtype=np.float32)
    s = int8_scale(x32)
    return int8_encode((x32 / s).astype(np.float32)), s  # fp32 division, IEEE RN


def dequantize_block(codes: np.ndarray, scale: float) -> np.ndarray:
    """x_hat = code * scale, in float64 (exact product)."""
    return np.asarray(codes, dtype=np.int8).astype(np.float64) * np.float64(np.float32(scale))


def quantize_chunk_bhld(x_blhd: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantise a token-major chunk ``[B, Lc, H, D]`` per (batch, head).

    Returns codes ``[B, H, Lc, D]`` int8 (head-major, like a ring slot) and
    scales ``[B, H]`` fp32."""
    x = np.transpose(np.asarray(x_blhd, dtype=np.float32), (0, 2, 1, 3))
    B, H = x.shape[:2]
    codes = np.empty(x.shape, dtype=np.int8)
    scales = np.empty((B, H), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            codes[b, h], scales[b, h] = quantize_block(x[b, h])
    return codes, scales
