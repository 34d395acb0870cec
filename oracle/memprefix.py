"""Block-causal attention behind a variable-length memory prefix -- oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).  float64, one library
matmul per product, the explicit token mask written out below.

Source: "WorldPlay2: Extending Real-Time Interactive World Models in Control
and Horizon" -- section 核心方法 (the history is summarised into a memory
m = [x_sink; x_cmp; x_tmp] that conditions the next chunk), section
方法步骤详情, training stage (3) (teacher forcing with a causal mask turns the
model into a chunk-level autoregressive one; the variable-length memory is
padded and the masked attention run with FlexAttention), and Figure 3 (causal
attention mask for compressed memory training).

Reading (the pages give the mask only as a figure; this is the plainest
reading consistent with the text):

* Each sample b is a sequence of L tokens: a memory prefix of ``mem_pad``
  positions, of which the first ``mem_len[b]`` are real and the rest padding,
  followed by target tokens in chunks of ``chunk_tokens`` (target token t
  belongs to chunk (t - mem_pad) // chunk_tokens).
* A real memory query sees every real memory key (the memory is one
  bidirectional block, like a sink chunk).
* A target query in chunk c sees every real memory key and the target keys of
  chunks c - W .. c (the block-causal rule of the training stage).
* Padding sees nothing and is seen by nothing: a padded query row has no
  visible key, so O = 0 and LSE = -inf there (the convention of
  ``attention.masked_attention``), and its gradients are zero.
"""

from __future__ import annotations

import numpy as np

from .attention import masked_attention


def memory_prefix_visibility(q_tok, k_tok, mem_pad: int, mem_len: int, chunk_tokens: int,
                             window: int) -> np.ndarray:
    """Mask ``[nq, nk]`` between query tokens ``q_tok`` and key tokens
    ``k_tok`` (token indices in one sample of the sequence)."""
    qt = np.asarray(q_tok, dtype=np.int64)[:, None]
    kt = np.asarray(k_tok, dtype=np.int64)[None, :]
    M, P, Lc, W = int(mem_pad), int(mem_len), int(chunk_tokens), int(window)
    q_mem_real = qt < P
    q_target = qt >= M
    k_mem_real = kt < P
    k_target = kt >= M
    d = (qt - M) // Lc - (kt - M) // Lc
    sees_memory = (q_mem_real | q_target) & k_mem_real
    sees_chunk = q_target & k_target & (d >= 0) & (d <= W)
    return sees_memory | sees_chunk


def memory_prefix_attention(q_blhd, k_blhd, v_blhd, mem_pad: int, mem_len, chunk_tokens: int, window: int,
                            scale: float, rows=None, heads=None, batches=None):
    """Forward over token-major ``[B, L, H, D]`` inputs; ``mem_len`` has one
    entry per sample.  Returns (O ``[nb, nh, nrows, D]``, LSE
    ``[nb, nh, nrows]``) for the selected rows / heads / batches."""
    q, k, v = np.asarray(q_blhd), np.asarray(k_blhd), np.asarray(v_blhd)
    B, L, H, _ = q.shape
    rows = np.arange(L) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = range(H) if heads is None else list(heads)
    batches = range(B) if batches is None else list(batches)
    O = np.empty((len(batches), len(heads), len(rows), v.shape[3]), dtype=np.float64)
    LSE = np.empty((len(batches), len(heads), len(rows)), dtype=np.float64)
    for bi, b in enumerate(batches):
        mask = memory_prefix_visibility(rows, np.arange(L), mem_pad, int(mem_len[b]), chunk_tokens, window)
        for hi, h in enumerate(heads):
            O[bi, hi], LSE[bi, hi] = masked_attention(np.asarray(q[b, rows, h], dtype=np.float64),
                                                      np.asarray(k[b, :, h], dtype=np.float64),
                                                      np.asarray(v[b, :, h], dtype=np.float64), mask, scale)
    return O, LSE


def _grad_head(q, k, v, do, mask, scale):
    """Gradients of one head under an explicit mask; rows with no visible key
    contribute nothing.  Same formulas as ``backward.block_causal_attention_
    backward``: dV = P^T dO, dS = P * (dO V^T - delta), dQ = scale dS K,
    dK = scale dS^T Q, delta = rowsum(dO * O)."""
    s = np.where(mask, scale * (q @ k.T), -np.inf)
    any_visible = mask.any(axis=1, keepdims=True)
    m = np.where(any_visible, np.max(s, axis=1, keepdims=True), 0.0)
    e = np.where(mask, np.exp(np.where(mask, s, 0.0) - m), 0.0)
    p = e / np.where(any_visible, e.sum(axis=1, keepdims=True), 1.0)
    o = p @ v
    delta = np.sum(do * o, axis=1, keepdims=True)
    ds = p * (do @ v.T - delta)
    dabs = np.sum(np.abs(do * o), axis=1, keepdims=True)
    grads = (scale * (ds @ k), scale * (ds.T @ q), p.T @ do)
    bounds = (scale * (np.abs(ds) @ np.abs(k) + dabs * (p @ np.abs(k))),
              scale * (np.abs(ds).T @ np.abs(q) + p.T @ (dabs * np.abs(q))),
              p.T @ np.abs(do))
    return grads, bounds


def memory_prefix_attention_backward(q_blhd, k_blhd, v_blhd, do_blhd, mem_pad: int, mem_len, chunk_tokens: int,
                                     window: int, scale: float):
    """(dQ, dK, dV) token-major ``[B, L, H, D]`` float64 and their per-element
    error scales (sums of absolute products, as in the block-causal gradient
    oracle)."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q_blhd, k_blhd, v_blhd, do_blhd))
    B, L, H, _ = q.shape
    out = [np.zeros_like(q) for _ in range(3)]
    bnd = [np.zeros_like(q) for _ in range(3)]
    tok = np.arange(L)
    for b in range(B):
        mask = memory_prefix_visibility(tok, tok, mem_pad, int(mem_len[b]), chunk_tokens, window)
        for h in range(H):
            g, e = _grad_head(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], mask, scale)
            for i in range(3):
                out[i][b, :, h] = g[i]
                bnd[i][b, :, h] = e[i]
    return tuple(out), tuple(bnd)
