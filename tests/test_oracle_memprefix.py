"""Pins of the memory-prefix attention oracle (``oracle/memprefix.py``)
against things it does not compute itself: a mask drawn by hand from the
reading of the WorldPlay2 causal-memory mask (Figure 3), the block-causal
oracle when there is no memory, PyTorch's scaled_dot_product_attention and
autograd in float64 with the same mask, finite differences, and invariances
of the padding."""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import memprefix as OM

# memory of 3 positions (2 real, 1 padding), then 3 target chunks of 2 tokens,
# window 1.  Rows: query tokens 0..8, columns: key tokens 0..8.
_HAND_MASK = np.array([
    # k: 0  1  2  3  4  5  6  7  8
    [1, 1, 0, 0, 0, 0, 0, 0, 0],  # q0 memory (real)
    [1, 1, 0, 0, 0, 0, 0, 0, 0],  # q1 memory (real)
    [0, 0, 0, 0, 0, 0, 0, 0, 0],  # q2 memory padding
    [1, 1, 0, 1, 1, 0, 0, 0, 0],  # q3 chunk 0
    [1, 1, 0, 1, 1, 0, 0, 0, 0],  # q4 chunk 0
    [1, 1, 0, 1, 1, 1, 1, 0, 0],  # q5 chunk 1
    [1, 1, 0, 1, 1, 1, 1, 0, 0],  # q6 chunk 1
    [1, 1, 0, 0, 0, 1, 1, 1, 1],  # q7 chunk 2 (chunk 0 has left the window)
    [1, 1, 0, 0, 0, 1, 1, 1, 1],  # q8 chunk 2
], dtype=bool)


def _inputs(B, L, H, D, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, L, H, D)) for _ in range(4)]


def test_mask_drawn_by_hand():
    t = np.arange(9)
    np.testing.assert_array_equal(OM.memory_prefix_visibility(t, t, 3, 2, 2, 1), _HAND_MASK)


def test_no_memory_is_block_causal():
    q, k, v, _ = _inputs(2, 70, 2, 8, 1)
    o, l = OM.memory_prefix_attention(q, k, v, 0, [0, 0], 16, 2, 0.4)
    o2, l2 = OA.block_causal_attention(q, k, v, 16, 2, 0.4)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("M,lens,Lc,W", [(40, (40, 17), 16, 2), (33, (0, 5), 10, 1), (7, (3, 7), 50, 0)])
def test_matches_torch_sdpa(M, lens, Lc, W):
    B, L, H, D = 2, 150, 2, 16
    q, k, v, _ = _inputs(B, L, H, D, 2)
    scale = 0.3
    o, l = OM.memory_prefix_attention(q, k, v, M, lens, Lc, W, scale)
    for b in range(B):
        t = torch.arange(L)
        tq = t[:, None]
        tk = t[None, :]
        # the reading written with torch ops on token indices, row by row
        real = lens[b]
        mem_q = tq < real
        tgt_q = tq >= M
        ch_q = torch.div(tq - M, Lc, rounding_mode="floor")
        ch_k = torch.div(tk - M, Lc, rounding_mode="floor")
        mask = ((mem_q | tgt_q) & (tk < real)) | (tgt_q & (tk >= M) & (ch_q - ch_k >= 0) & (ch_q - ch_k <= W))
        for h in range(H):
            qt, kt, vt = (torch.from_numpy(x[b, :, h]) for x in (q, k, v))
            rows = mask.any(dim=1)
            ref = torch.nn.functional.scaled_dot_product_attention(qt[rows][None], kt[None], vt[None],
                                                                   attn_mask=mask[rows][None], scale=scale)[0]
            np.testing.assert_allclose(o[b, h][rows.numpy()], ref.numpy(), rtol=0, atol=1e-12)
            assert np.all(o[b, h][~rows.numpy()] == 0.0)
            assert np.all(np.isneginf(l[b, h][~rows.numpy()]))
            s = scale * (qt[rows] @ kt.T)
            lse = torch.logsumexp(s.masked_fill(~mask[rows], -torch.inf), dim=1)
            np.testing.assert_allclose(l[b, h][rows.numpy()], lse.numpy(), rtol=0, atol=1e-12)


def test_padding_is_inert():
    """Changing the padded positions' keys and values changes no output of a
    real row; a real memory row equals plain attention over the real memory."""
    B, L, H, D, M = 1, 90, 1, 8, 30
    q, k, v, _ = _inputs(B, L, H, D, 3)
    o, _ = OM.memory_prefix_attention(q, k, v, M, [12], 20, 1, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[:, 12:M] = 100.0
    v2[:, 12:M] = -50.0
    o2, _ = OM.memory_prefix_attention(q, k2, v2, M, [12], 20, 1, 0.5)
    real = np.r_[0:12, M:L]
    np.testing.assert_array_equal(o[0, 0][real], o2[0, 0][real])
    qt, kt, vt = (torch.from_numpy(x[0, :12, 0]) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None], scale=0.5)[0]
    np.testing.assert_allclose(o[0, 0][:12], ref.numpy(), rtol=0, atol=1e-12)


def test_gradients_match_torch_autograd():
    B, L, H, D, M, Lc, W, scale = 2, 96, 2, 8, 24, 16, 2, 0.35
    lens = (24, 9)
    q, k, v, do = _inputs(B, L, H, D, 4)
    (dq, dk, dv), _ = OM.memory_prefix_attention_backward(q, k, v, do, M, lens, Lc, W, scale)
    for b in range(B):
        mask = torch.from_numpy(OM.memory_prefix_visibility(np.arange(L), np.arange(L), M, lens[b], Lc, W))
        rows = mask.any(dim=1)
        for h in range(H):
            qt, kt, vt = (torch.from_numpy(x[b, :, h]).requires_grad_(True) for x in (q, k, v))
            s = (scale * qt @ kt.T).masked_fill(~mask, -torch.inf)
            p = torch.softmax(s[rows], dim=1)
            o = p @ vt
            (o * torch.from_numpy(do[b, :, h])[rows]).sum().backward()
            np.testing.assert_allclose(dq[b, :, h], qt.grad.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(dk[b, :, h], kt.grad.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(dv[b, :, h], vt.grad.numpy(), rtol=0, atol=1e-12)


def test_gradients_finite_differences():
    """Central differences of sum(O * dO) through the forward oracle."""
    B, L, H, D, M, Lc, W, scale = 1, 20, 1, 4, 6, 5, 1, 0.7
    lens = (4,)
    q, k, v, do = _inputs(B, L, H, D, 5)
    (dq, dk, dv), _ = OM.memory_prefix_attention_backward(q, k, v, do, M, lens, Lc, W, scale)

    def loss(q_, k_, v_):
        o, _ = OM.memory_prefix_attention(q_, k_, v_, M, lens, Lc, W, scale)
        return float(np.sum(o[0, 0] * do[0, :, 0]))

    eps = 1e-6
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        for (t, d) in ((0, 1), (3, 2), (5, 0), (6, 3), (13, 1), (19, 2)):
            xs = [q, k, v]
            plus = [x.copy() for x in xs]
            minus = [x.copy() for x in xs]
            plus[which][0, t, 0, d] += eps
            minus[which][0, t, 0, d] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - grad[0, t, 0, d]) <= 1e-7 + 1e-6 * abs(fd), (which, t, d, fd, grad[0, t, 0, d])
    # padded positions (4, 5) get no gradient at all
    for g in (dq, dk, dv):
        assert np.all(g[0, 4:6] == 0.0)
