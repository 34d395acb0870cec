"""Attention with E4M3 tensor-core products (Q and P in 8 bits) -- oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).  float64 on exact
dequantised values, one library matmul per product.

Source: "Matrix-Game 4.0: Harnessing Video Models for Real-Time Playable Game
Worlds", sections 前置知识 / FP8 量化与 CUDA Graph (attention and linear layers
computed in FP8) and 技术新颖性 (8-bit keys and values per KV interval).  The
pages do not say how the query and the probabilities enter the 8-bit product.
Reading:

* Q: each query row of one head is quantised on its own with the absmax rule
  of the cache (``fp8.quantize_block`` over the row's D values): one fp32
  scale amax/448 per row, codes rounded to nearest even with satfinite, the
  division in fp32.  This decision is the same on both sides, so the oracle
  uses the kernel's q-hat exactly.
* K, V: the cache's dequantised values (codes x per-(head, chunk) scale).
* P: the probabilities are rounded to E4M3 before the P V product.  Their
  exact values depend on the device's exponential, so the oracle does not
  replay that rounding; it returns the exact result on (q-hat, k-hat, v-hat)
  and a per-element bound on what rounding P can change.

The bound.  A key j of the row is rounded in the form
P'_j = P_j * r_j * 2^(g + delta), where P_j = exp(s_j - max) <= 1,
r_j = vs_j / vs_ref <= 1 is the key's V scale relative to the largest V scale
of the visible keys (the V scales are applied before the rounding so that the
product uses the codes as stored), g is a fixed gain that lifts the values
out of the subnormal range (the kernel uses g = 3 with a running-max slack
of at most 2^5.75, so P' <= 2^8.75 < 448), and delta >= 0 accounts for a running
maximum that has not yet caught up (the values are then larger, never
smaller).  E4M3 rounding to nearest changes a value by at most 2^-4 of itself
when it is normal (>= 2^-6) and by at most 2^-10 (half the subnormal spacing
2^-9) -- and never by more than the value, which can round to 0 -- below
that.  In units of P_j:

    e_j = 2^-4 P_j                          if P_j r_j 2^g >= 2^-6
          min(P_j, 2^-10 / (r_j 2^g))       otherwise

and O_i = sum_j P_ij v_j / l_i (l_i = sum_j P_ij, kept in fp32 from the
unrounded values) moves by at most  bound_i = sum_j e_ij |v_j| / l_i  per
output column.

The typical size.  Modelling each rounding error as uniform over one E4M3
spacing u_j of P'_j (spacing 2^(floor(log2 P') - 3) when normal, 2^-9 below
2^-6; in units of P divided by r_j 2^g) and independent across keys, the
error of O_id has standard deviation
sigma_id = sqrt(sum_j (u_j^2 / 12) v_jd^2) / l_i, and its mean magnitude is
about sqrt(2 / pi) sigma_id.
"""

from __future__ import annotations

import numpy as np

from .fp8 import dequantize_block, quantize_block


def quantize_rows(q: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-row E4M3 quantisation of ``q [rows, D]``: returns (q_hat float64
    [rows, D], scales fp32 [rows])."""
    q = np.asarray(q, dtype=np.float32)
    out = np.empty(q.shape, dtype=np.float64)
    sc = np.empty(q.shape[0], dtype=np.float32)
    for i in range(q.shape[0]):
        codes, s = quantize_block(q[i:i + 1])
        out[i] = dequantize_block(codes, s)[0]
        sc[i] = s
    return out, sc


P_GAIN_LOG2 = 3  # g of the module docstring


def p_rounding_error(p: np.ndarray, r: np.ndarray, gain_log2: int = P_GAIN_LOG2) -> np.ndarray:
    """e_ij of the module docstring for probabilities ``p [n, Nk]`` (max 1 per
    row), relative V scales ``r [Nk]`` and gain 2^gain_log2."""
    p = np.asarray(p, dtype=np.float64)
    rg = np.asarray(r, dtype=np.float64)[None, :] * 2.0 ** gain_log2
    normal = p * rg >= 2.0 ** -6
    return np.where(normal, 2.0 ** -4 * p, np.minimum(p, 2.0 ** -10 / rg))


def p_rounding_spacing(p: np.ndarray, r: np.ndarray, gain_log2: int = P_GAIN_LOG2) -> np.ndarray:
    """u_j of the module docstring (E4M3 spacing at P' = P r 2^g, in units of
    P) for probabilities ``p [n, Nk]`` and relative V scales ``r [Nk]``."""
    p = np.asarray(p, dtype=np.float64)
    rg = np.asarray(r, dtype=np.float64)[None, :] * 2.0 ** gain_log2
    x = p * rg
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -6)))
    return 2.0 ** (e - 3) / rg


def rounding_sigma(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, mask: np.ndarray, scale: float,
                   v_scale_key: np.ndarray, gain_log2: int = P_GAIN_LOG2) -> np.ndarray:
    """sigma ``[Lq, D]`` of the module docstring for the inputs of
    ``head_attention``."""
    q_hat, _ = quantize_rows(q)
    k = np.asarray(k_hat, dtype=np.float64)
    v = np.asarray(v_hat, dtype=np.float64)
    mask = np.asarray(mask, dtype=bool)
    vs = np.asarray(v_scale_key, dtype=np.float64)
    s = np.where(mask, float(scale) * (q_hat @ k.T), -np.inf)
    p = np.where(mask, np.exp(s - np.max(s, axis=1, keepdims=True)), 0.0)
    l = p.sum(axis=1, keepdims=True)
    vs_ref = np.max(np.where(mask.any(axis=0), vs, 0.0))
    r = np.where(vs > 0, vs / vs_ref, 1.0)
    u = np.where(mask, p_rounding_spacing(p, r, gain_log2), 0.0)
    return np.sqrt((u * u / 12.0) @ (v * v)) / l


def head_attention(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, mask: np.ndarray, scale: float,
                   v_scale_key: np.ndarray, gain_log2: int = P_GAIN_LOG2):
    """One head: q ``[Lq, D]`` (the bf16 queries, quantised here per row),
    k_hat, v_hat ``[Nk, D]`` dequantised cache rows, mask ``[Lq, Nk]`` (every
    row sees at least one key), v_scale_key ``[Nk]`` the V scale of each key's
    chunk.  Returns (O ``[Lq, D]``, LSE ``[Lq]``, bound ``[Lq, D]``) in float64."""
    q_hat, _ = quantize_rows(q)
    k = np.asarray(k_hat, dtype=np.float64)
    v = np.asarray(v_hat, dtype=np.float64)
    mask = np.asarray(mask, dtype=bool)
    vs = np.asarray(v_scale_key, dtype=np.float64)
    s = np.where(mask, float(scale) * (q_hat @ k.T), -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    p = np.where(mask, np.exp(s - m), 0.0)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ v) / l
    lse = (m + np.log(l))[:, 0]
    # relative V scales over the keys the rows see
    vs_ref = np.max(np.where(mask.any(axis=0), vs, 0.0))
    r = np.where(vs > 0, vs / vs_ref, 1.0)
    e = np.where(mask, p_rounding_error(p, r, gain_log2), 0.0)
    bound = (e @ np.abs(v)) / l
    return o, lse, bound
