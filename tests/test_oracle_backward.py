"""Pins of the attention-gradient oracle (``oracle/backward.py``) against
things it does not compute itself: central finite differences of the loss
sum(O * dO) through the forward oracle, PyTorch autograd in float64 with the
same mask, and structural facts (keys no query sees get zero gradient; the
value gradient of a chunk-local mask is block diagonal)."""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import backward as OB


def _inputs(B, L, H, D, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, L, H, D)) for _ in range(4)]


def _loss(q, k, v, do, Lc, W, scale):
    o, _ = OA.block_causal_attention(q, k, v, Lc, W, scale)  # [B, H, L, D]
    return float(np.sum(o * np.transpose(do, (0, 2, 1, 3))))


def test_finite_differences():
    q, k, v, do = _inputs(1, 6, 2, 3, 1)
    Lc, W, scale = 2, 1, 0.7
    grads = OB.block_causal_attention_backward(q, k, v, do, Lc, W, scale)
    eps = 1e-6
    rng = np.random.default_rng(2)
    for which, (x, g) in enumerate(zip((q, k, v), grads)):
        for _ in range(6):
            idx = tuple(rng.integers(0, n) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num = (_loss(*args_p, do, Lc, W, scale) - _loss(*args_m, do, Lc, W, scale)) / (2 * eps)
            assert abs(num - g[idx]) <= 1e-6 * (1 + abs(num)), (which, idx, num, g[idx])


def test_matches_torch_autograd():
    q, k, v, do = _inputs(2, 10, 3, 4, 3)
    Lc, W, scale = 3, 1, 0.5
    dq, dk, dv = OB.block_causal_attention_backward(q, k, v, do, Lc, W, scale)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    chunk = torch.arange(10) // Lc
    diff = chunk[:, None] - chunk[None, :]
    allowed = (diff >= 0) & (diff <= W)
    s = scale * torch.einsum("blhd,bmhd->bhlm", tq, tk)
    s = s.masked_fill(~allowed, float("-inf"))
    o = torch.einsum("bhlm,bmhd->blhd", torch.softmax(s, dim=-1), tv)
    (o * torch.tensor(do)).sum().backward()
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-12)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-12)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_structure_and_bounds():
    q, k, v, do = _inputs(1, 8, 1, 4, 4)
    # window 0: each chunk attends only to itself -> gradients stay inside chunks
    (dq, dk, dv), (bq, bk, bv) = OB.block_causal_attention_backward(q, k, v, do, 4, 0, 1.0, abs_bounds=True)
    dq2, dk2, dv2 = OB.block_causal_attention_backward(q[:, :4], k[:, :4], v[:, :4], do[:, :4], 4, 0, 1.0)
    assert np.allclose(dq[:, :4], dq2) and np.allclose(dk[:, :4], dk2) and np.allclose(dv[:, :4], dv2)
    assert np.all(np.abs(dq) <= bq + 1e-12) and np.all(np.abs(dk) <= bk + 1e-12) and np.all(np.abs(dv) <= bv + 1e-12)
    # every query's probabilities sum to 1, so the value gradients of all keys
    # sum to the sum of the output gradients
    assert np.allclose(dv.sum(axis=1), do.sum(axis=1))


def test_sampled_rows_equal_full():
    """The row-restricted form returns the full form's rows (ragged last
    chunk, window 2, rows at chunk edges and inside)."""
    B, L, H, D, Lc, W = 2, 340, 2, 16, 64, 2
    q, k, v, do = _inputs(B, L, H, D, 11)
    (fq, fk, fv), (gq, gk, gv) = OB.block_causal_attention_backward(q, k, v, do, Lc, W, 0.3, abs_bounds=True)
    qr = np.array([0, 63, 64, 200, 339])
    kr = np.array([1, 64, 127, 128, 300, 339])
    for b, h in ((0, 1), (1, 0)):
        (dq, dk, dv), (bq, bk, bv) = OB.block_causal_attention_backward_rows(q, k, v, do, Lc, W, 0.3, b, h, qr, kr)
        np.testing.assert_allclose(dq, fq[b, qr, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dk, fk[b, kr, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dv, fv[b, kr, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(bq, gq[b, qr, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(bk, gk[b, kr, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(bv, gv[b, kr, h], rtol=1e-12, atol=1e-13)
