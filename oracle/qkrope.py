"""Q/K RMS normalisation and rotary position embedding of one chunk -- oracle
(test infrastructure).

Not for the product path; see the package docstring.

The pages name the fused step but not its formulas: "WorldPlay2: Extending
Real-Time Interactive World Models in Control and Horizon", section 方法步骤
详情 (inference: QKRoPE and QKV fusion), and "Matrix-Game 4.0: Harnessing
Video Models for Real-Time Playable Game Worlds", section 实验结果 (a fused
RoPE kernel on the causal Wan DiT).  The reading used here is the plain one
for a Wan-style video DiT:

* RMSNorm of q (and of k) over the token's whole hidden vector of H*D values:
  y = x / sqrt(mean(x^2) + eps) * gamma, gamma of length H*D (1 when absent),
  eps = 1e-6.
* Rotary embedding per head on interleaved pairs (2i, 2i+1), rotated by the
  angle pos * theta_i with theta_i = base^(-2i / band) inside each band:
  the head dimension is split into three bands (frame, height, width) of
  Dt + Dh + Dw = D dimensions (even), each band rotated by its own position
  coordinate.  Token t of chunk c sits at frame c * F + t // (Hp * Wp), row
  (t // Wp) % Hp and column t % Wp of a latent grid of F frames x Hp x Wp
  patches per chunk (Lc = F * Hp * Wp).  Dh = Dw = 0 and Hp = Wp = 1 give the
  classic one-dimensional rotary embedding over the token index.
* V passes through unchanged.

Everything is computed in float64 on the bf16 inputs.
"""

from __future__ import annotations

import numpy as np

EPS = 1e-6
BASE = 10000.0


def rms_norm(x_blhd: np.ndarray, gamma=None, eps: float = EPS) -> np.ndarray:
    """RMSNorm over H*D per token of a [B, L, H, D] array (float64)."""
    x = np.asarray(x_blhd, dtype=np.float64)
    B, L, H, D = x.shape
    flat = x.reshape(B, L, H * D)
    inv = 1.0 / np.sqrt(np.mean(flat * flat, axis=-1, keepdims=True) + eps)
    y = flat * inv
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64).reshape(1, 1, H * D)
    return y.reshape(B, L, H, D)


def positions(chunk: int, Lc: int, grid) -> np.ndarray:
    """[Lc, 3] (frame, row, column) coordinates of the chunk's tokens."""
    F, Hp, Wp = grid
    assert F * Hp * Wp == Lc
    t = np.arange(Lc)
    return np.stack([chunk * F + t // (Hp * Wp), (t // Wp) % Hp, t % Wp], axis=1).astype(np.float64)


def angles(pos: np.ndarray, bands, base: float = BASE) -> np.ndarray:
    """[L, D/2] rotation angle of each (token, pair) for band sizes (Dt, Dh, Dw)."""
    cols = []
    for axis, band in enumerate(bands):
        if band == 0:
            continue
        i = np.arange(band // 2, dtype=np.float64)
        theta = base ** (-2.0 * i / band)
        cols.append(pos[:, axis:axis + 1] * theta[None, :])
    return np.concatenate(cols, axis=1)


def rope(x_blhd: np.ndarray, ang_ld2: np.ndarray) -> np.ndarray:
    """Rotate interleaved pairs of every head of [B, L, H, D] by [L, D/2] angles."""
    x = np.asarray(x_blhd, dtype=np.float64)
    c = np.cos(ang_ld2)[None, :, None, :]
    s = np.sin(ang_ld2)[None, :, None, :]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def qk_norm_rope(q_blhd, k_blhd, chunk: int, grid, bands, gamma_q=None, gamma_k=None, base: float = BASE):
    """(q', k') of one chunk: RMSNorm then rotary embedding."""
    Lc = np.asarray(q_blhd).shape[1]
    ang = angles(positions(chunk, Lc, grid), bands, base)
    return rope(rms_norm(q_blhd, gamma_q), ang), rope(rms_norm(k_blhd, gamma_k), ang)
