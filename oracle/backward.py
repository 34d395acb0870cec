"""Gradients of block-causal attention -- oracle (test infrastructure).

Not for the product path; see the package docstring.

The pages train the streaming model with a block-causal mask ("WanToFight:
Real-Time Generative Game Engine for Multi-Player Combat Interaction",
section 训练流程 / Stage 2: the dense mask is replaced by a block-causal one;
"WorldPlay2", Figure 3 and section 方法步骤详情: teacher forcing with a causal
chunk mask).  Training needs the gradients of the same attention.  They are
the plain derivatives of O = softmax(scale * Q K^T + mask) V for a loss whose
gradient with respect to O is dO:

    P   = softmax over visible keys of scale * q_i . k_j
    dV  = P^T dO
    dP  = dO V^T
    dS  = P * (dP - delta),  delta_i = sum_j P_ij dP_ij = sum_d dO_id O_id
    dQ  = scale * dS K
    dK  = scale * dS^T Q

computed in float64 with the explicit token mask (query i sees key j iff
0 <= chunk(i) - chunk(j) <= window).  ``abs_bounds`` also returns, for every
output element, the scale of the rounding error of a finite-precision
evaluation: the sum of the absolute values of the products it adds up, plus
(dQ, dK) the sensitivity to an error in delta of relative size 1 --
scale * sum_j P_ij * (sum_d |dO_id O_id|) * |K_jd| (dQ) and likewise with Q
(dK) -- since delta is itself a sum of products.
"""

from __future__ import annotations

import numpy as np

from .attention import chunk_visibility


def _head(q, k, v, do, mask, scale):
    """One head: q, k, v, do [L, D] float64, mask [L, L] bool."""
    s = scale * (q @ k.T)
    s = np.where(mask, s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    e = np.where(mask, np.exp(s - m), 0.0)
    p = e / e.sum(axis=1, keepdims=True)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    delta = np.sum(do * o, axis=1, keepdims=True)
    ds = p * (dp - delta)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, p, ds


def block_causal_attention_backward(q_blhd, k_blhd, v_blhd, do_blhd, chunk_tokens: int, window: int,
                                    scale: float, abs_bounds: bool = False):
    """(dQ, dK, dV) token-major [B, L, H, D] float64; with ``abs_bounds`` also
    (|dQ|, |dK|, |dV|) bounds: sum_j |a_j| |b_j| of each output's products."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q_blhd, k_blhd, v_blhd, do_blhd))
    B, L, H, D = q.shape
    chunk = np.arange(L) // int(chunk_tokens)
    mask = chunk_visibility(chunk, chunk, window)
    out = [np.zeros_like(q) for _ in range(3)]
    bnd = [np.zeros_like(q) for _ in range(3)] if abs_bounds else None
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
            dq, dk, dv, p, ds = _head(qh, kh, vh, doh, mask, scale)
            out[0][b, :, h], out[1][b, :, h], out[2][b, :, h] = dq, dk, dv
            if abs_bounds:
                o = p @ vh
                dabs = np.sum(np.abs(doh * o), axis=1, keepdims=True)  # scale of delta's rounding
                bnd[0][b, :, h] = scale * (np.abs(ds) @ np.abs(kh) + dabs * (p @ np.abs(kh)))
                bnd[1][b, :, h] = scale * (np.abs(ds).T @ np.abs(qh) + p.T @ (dabs * np.abs(qh)))
                bnd[2][b, :, h] = np.abs(p).T @ np.abs(doh)
    return (tuple(out), tuple(bnd)) if abs_bounds else tuple(out)


def block_causal_attention_backward_rows(q_blhd, k_blhd, v_blhd, do_blhd, chunk_tokens: int, window: int,
                                         scale: float, b: int, h: int, q_rows, k_rows):
    """The same gradients for one (batch, head), only at sampled rows: dQ at
    ``q_rows`` and dK, dV at ``k_rows`` (float64 [n, D] each, plus the error
    scales of ``block_causal_attention_backward``).  Every query that sees a
    sampled key contributes its full softmax row, computed chunk by chunk
    over the keys that chunk sees; no other reordering."""
    q, k, v, do = (np.asarray(x[b, :, h], dtype=np.float64) for x in (q_blhd, k_blhd, v_blhd, do_blhd))
    L, D = q.shape
    Lc, W = int(chunk_tokens), int(window)
    q_rows, k_rows = np.asarray(q_rows), np.asarray(k_rows)
    nchunks = (L + Lc - 1) // Lc
    need = set((q_rows // Lc).tolist())
    for c in set((k_rows // Lc).tolist()):
        need.update(range(c, min(nchunks, c + W + 1)))
    dq, bq = np.zeros((len(q_rows), D)), np.zeros((len(q_rows), D))
    dk, bk = np.zeros((len(k_rows), D)), np.zeros((len(k_rows), D))
    dv, bv = np.zeros((len(k_rows), D)), np.zeros((len(k_rows), D))
    for c in sorted(need):
        qs = np.arange(c * Lc, min(L, (c + 1) * Lc))
        ks = np.arange(max(0, c - W) * Lc, min(L, (c + 1) * Lc))  # keys of chunks c - W .. c
        s = scale * (q[qs] @ k[ks].T)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        p = e / e.sum(axis=1, keepdims=True)
        o = p @ v[ks]
        delta = np.sum(do[qs] * o, axis=1, keepdims=True)
        ds = p * (do[qs] @ v[ks].T - delta)
        dabs = np.sum(np.abs(do[qs] * o), axis=1, keepdims=True)
        sel = np.nonzero((q_rows // Lc) == c)[0]
        if sel.size:
            li = q_rows[sel] - c * Lc
            dq[sel] = scale * (ds[li] @ k[ks])
            bq[sel] = scale * (np.abs(ds[li]) @ np.abs(k[ks]) + dabs[li] * (p[li] @ np.abs(k[ks])))
        kin = np.nonzero((k_rows >= ks[0]) & (k_rows <= ks[-1]))[0]
        if kin.size:
            lj = k_rows[kin] - ks[0]
            dv[kin] += p[:, lj].T @ do[qs]
            bv[kin] += p[:, lj].T @ np.abs(do[qs])
            dk[kin] += scale * (ds[:, lj].T @ q[qs])
            bk[kin] += scale * (np.abs(ds[:, lj]).T @ np.abs(q[qs]) + p[:, lj].T @ (dabs * np.abs(q[qs])))
    return (dq, dk, dv), (bq, bk, bv)
