"""Pins for the oracle's attention arithmetic (CPU only).

Each test checks the oracle against something other than itself: brute force
on tiny inputs written with scalar loops, a hand-computed worked example, the
PyTorch scaled-dot-product-attention routine in fp64 for the cases that reduce
to plain attention, closed forms (Q = 0, identical V rows) and invariants
(row sums, key permutation, split-and-merge).  A dropped term, a wrong sign or
index or a transposed operand in the oracle fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle.ring import ListRing, RingError

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute(q, k, v, mask, scale):
    """Scalar-loop attention, fp64, math.exp only."""
    Lq, Nk, Dv = q.shape[0], k.shape[0], v.shape[1]
    O = np.zeros((Lq, Dv))
    L = np.zeros(Lq)
    for i in range(Lq):
        s = []
        for j in range(Nk):
            if mask[i, j]:
                acc = 0.0
                for d in range(q.shape[1]):
                    acc += float(q[i, d]) * float(k[j, d])
                s.append((j, scale * acc))
        mx = max(x for _, x in s)
        den = sum(math.exp(x - mx) for _, x in s)
        for j, x in s:
            p = math.exp(x - mx) / den
            for d in range(Dv):
                O[i, d] += p * float(v[j, d])
        L[i] = mx + math.log(den)
    return O, L


def _sdpa(q, k, v, scale):
    """torch SDPA in fp64 on [L, D] inputs; LSE from torch.logsumexp."""
    tq, tk, tv = (torch.as_tensor(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], scale=scale)[0]
    lse = torch.logsumexp(scale * tq @ tk.T, dim=-1)
    return o.numpy(), lse.numpy()


def test_two_key_worked_example():
    vals = {}
    with open(os.path.join(GOLDEN, "two_key_attention.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, rest = line.split(None, 1)
            vals[name] = rest.strip()
    scale = float(vals["scale"])
    q = np.array([[float(x) for x in vals["q"].split()]])
    k = np.array([[float(x) for x in r.split()] for r in vals["k"].split(";")])
    v = np.array([[float(x) for x in r.split()] for r in vals["v"].split(";")])
    mask = np.array([[bool(int(x)) for x in vals["mask"].split()]])
    o, lse = A.masked_attention(q, k, v, mask, scale)
    assert o[0, 0] == pytest.approx(float(vals["O0"]), abs=1e-15)
    assert o[0, 1] == pytest.approx(float(vals["O1"]), abs=1e-15)
    assert lse[0] == pytest.approx(float(vals["LSE"]), abs=1e-15)


@pytest.mark.parametrize("seed", range(6))
def test_masked_attention_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    Lq, Nk, D, Dv = rng.integers(1, 5), rng.integers(1, 9), rng.integers(1, 9), rng.integers(1, 6)
    q, k, v = rng.normal(size=(Lq, D)), rng.normal(size=(Nk, D)), rng.normal(size=(Nk, Dv))
    mask = rng.random((Lq, Nk)) < 0.7
    mask[:, rng.integers(0, Nk)] = True  # every row has a visible key
    scale = float(rng.uniform(0.1, 2.0))
    o, lse = A.masked_attention(q, k, v, mask, scale)
    ob, lb = _brute(q, k, v, mask, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-13)


def test_asymmetric_qk_roles():
    """Swapping q and k (a transposed product) must change the answer."""
    rng = np.random.default_rng(7)
    q, k, v = rng.normal(size=(3, 4)), rng.normal(size=(5, 4)), rng.normal(size=(5, 2))
    mask = np.ones((3, 5), bool)
    o, _ = A.masked_attention(q, k, v, mask, 0.5)
    ob, _ = _brute(q, k, v, mask, 0.5)
    np.testing.assert_allclose(o, ob, atol=1e-13)


def test_row_sums_and_masked_zero():
    """With V = identity, O is the probability matrix: rows sum to 1, masked
    entries are exactly 0."""
    rng = np.random.default_rng(3)
    Lq, Nk, D = 6, 11, 8
    q, k = rng.normal(size=(Lq, D)), rng.normal(size=(Nk, D))
    mask = rng.random((Lq, Nk)) < 0.5
    mask[:, 0] = True
    p, _ = A.masked_attention(q, k, np.eye(Nk), mask, 0.3)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(p[~mask] == 0.0)
    assert np.all(p[mask] > 0.0)


def test_q_zero_closed_form():
    rng = np.random.default_rng(4)
    Nk, D = 13, 8
    k, v = rng.normal(size=(Nk, D)), rng.normal(size=(Nk, 5))
    mask = np.zeros((2, Nk), bool)
    mask[0, [1, 4, 5, 9]] = True
    mask[1, :] = True
    o, lse = A.masked_attention(np.zeros((2, D)), k, v, mask, 0.7)
    np.testing.assert_allclose(o[0], v[[1, 4, 5, 9]].mean(axis=0), atol=1e-14)
    np.testing.assert_allclose(o[1], v.mean(axis=0), atol=1e-14)
    np.testing.assert_allclose(lse, [math.log(4), math.log(Nk)], atol=1e-14)


def test_identical_v_rows():
    rng = np.random.default_rng(5)
    row = rng.normal(size=7)
    v = np.tile(row, (9, 1))
    q, k = rng.normal(size=(4, 3)) * 5, rng.normal(size=(9, 3)) * 5
    mask = rng.random((4, 9)) < 0.6
    mask[:, 2] = True
    o, _ = A.masked_attention(q, k, v, mask, 1.0)
    np.testing.assert_allclose(o, np.tile(row, (4, 1)), atol=1e-13)


def test_key_permutation_invariance():
    rng = np.random.default_rng(6)
    q, k, v = rng.normal(size=(5, 8)), rng.normal(size=(17, 8)), rng.normal(size=(17, 8))
    mask = rng.random((5, 17)) < 0.6
    mask[:, 3] = True
    o, lse = A.masked_attention(q, k, v, mask, 0.4)
    perm = rng.permutation(17)
    o2, lse2 = A.masked_attention(q, k[perm], v[perm], mask[:, perm], 0.4)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)


@pytest.mark.parametrize("nsplit", [1, 2, 3, 7])
def test_split_merge_equivalence(nsplit):
    rng = np.random.default_rng(10 + nsplit)
    Lq, Nk, D = 4, 23, 8
    q, k, v = rng.normal(size=(Lq, D)) * 3, rng.normal(size=(Nk, D)), rng.normal(size=(Nk, D))
    mask = rng.random((Lq, Nk)) < 0.8
    mask[:, 0] = True
    o, lse = A.masked_attention(q, k, v, mask, 0.5)
    part = rng.integers(0, nsplit + 1, size=Nk)  # one extra label so a part can be empty
    po, pl = [], []
    for s in range(nsplit + 2):  # includes surely-empty parts
        sel = part == s
        m = mask & sel[None, :]
        a, b = A.masked_attention(q, k, v, m, 0.5)
        po.append(a); pl.append(b)
    om, lm = A.lse_merge(po, pl)
    np.testing.assert_allclose(om, o, atol=1e-12)
    np.testing.assert_allclose(lm, lse, atol=1e-12)


def test_lse_merge_all_empty():
    o, l = A.lse_merge([np.zeros((2, 3)), np.zeros((2, 3))], [np.full(2, -np.inf), np.full(2, -np.inf)])
    assert np.all(o == 0) and np.all(np.isneginf(l))


def _blhd_to_bhld(x):
    return np.transpose(np.asarray(x), (0, 2, 1, 3))


def _stream_setup(seed, B=1, H=2, Lc=3, D=4, chunks=5, R=2):
    rng = np.random.default_rng(seed)
    ks = [rng.normal(size=(B, H, Lc, D)) for _ in range(chunks)]
    vs = [rng.normal(size=(B, H, Lc, D)) for _ in range(chunks)]
    qs = [rng.normal(size=(B, H, Lc, D)) for _ in range(chunks)]
    return rng, ks, vs, qs


def test_single_chunk_equals_sdpa():
    """Chunk 0, no sink: plain bidirectional attention over the chunk."""
    rng, ks, vs, qs = _stream_setup(20, Lc=6, D=8)
    ring = ListRing(2)
    o, lse = A.streaming_chunk_attention(qs[0], ring, 0, ks[0], vs[0], 2, False, 0.35)
    for b in range(1):
        for h in range(2):
            so, sl = _sdpa(qs[0][b, h], ks[0][b, h], vs[0][b, h], 0.35)
            np.testing.assert_allclose(o[b, h], so, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], sl, atol=1e-12)


def test_full_window_equals_full_attention():
    """W >= c with a ring holding every chunk: attention over all streamed tokens."""
    rng, ks, vs, qs = _stream_setup(21, chunks=4, R=8)
    ring = ListRing(8)
    for c in range(3):
        ring.append(c, ks[c], vs[c])
    o, lse = A.streaming_chunk_attention(qs[3], ring, 3, ks[3], vs[3], 5, False, 0.5)
    kall = np.concatenate(ks[:4], axis=2)
    vall = np.concatenate(vs[:4], axis=2)
    for h in range(2):
        so, sl = _sdpa(qs[3][0, h], kall[0, h], vall[0, h], 0.5)
        np.testing.assert_allclose(o[0, h], so, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], sl, atol=1e-12)


def test_window_excludes_old_chunks_and_sink_included():
    """Streaming result equals SDPA over exactly sink + chunks c-W..c (slicing,
    not masking), for every chunk of a stream that wraps the ring."""
    rng, ks, vs, qs = _stream_setup(22, chunks=7, R=3)
    sk, sv = rng.normal(size=(1, 2, 3, 4)), rng.normal(size=(1, 2, 3, 4))
    ring = ListRing(3)
    ring.set_sink(sk, sv)
    W = 2
    for c in range(7):
        o, lse = A.streaming_chunk_attention(qs[c], ring, c, ks[c], vs[c], W, True, 0.6)
        lo = max(0, c - W)
        kk = np.concatenate([sk] + ks[lo:c + 1], axis=2)
        vv = np.concatenate([sv] + vs[lo:c + 1], axis=2)
        for h in range(2):
            so, sl = _sdpa(qs[c][0, h], kk[0, h], vv[0, h], 0.6)
            np.testing.assert_allclose(o[0, h], so, atol=1e-12)
            np.testing.assert_allclose(lse[0, h], sl, atol=1e-12)
        ring.append(c, ks[c], vs[c])


def test_current_chunk_in_ring_equals_passed_in():
    """Appending chunk c first and attending from the ring equals passing K_cur."""
    rng, ks, vs, qs = _stream_setup(23, chunks=6, R=4)
    r1, r2 = ListRing(4), ListRing(4)
    for c in range(6):
        o1, l1 = A.streaming_chunk_attention(qs[c], r1, c, ks[c], vs[c], 3, False, 0.5)
        r1.append(c, ks[c], vs[c])
        r2.append(c, ks[c], vs[c])
        o2, l2 = A.streaming_chunk_attention(qs[c], r2, c, None, None, 3, False, 0.5)
        np.testing.assert_allclose(o2, o1, atol=1e-12)
        np.testing.assert_allclose(l2, l1, atol=1e-12)


def test_missing_chunk_raises():
    rng, ks, vs, qs = _stream_setup(24, chunks=5, R=2)
    ring = ListRing(2)
    for c in range(4):
        ring.append(c, ks[c], vs[c])
    with pytest.raises(RingError):  # window 3 needs chunk 1, evicted
        A.streaming_chunk_attention(qs[4], ring, 4, ks[4], vs[4], 3, False, 0.5)
    with pytest.raises(RingError):  # no K_cur and chunk 4 not appended
        A.streaming_chunk_attention(qs[4], ring, 4, None, None, 1, False, 0.5)


def test_block_causal_equals_sliced_sdpa():
    rng = np.random.default_rng(30)
    B, nch, Lc, H, D, W = 2, 5, 3, 2, 4, 2
    q, k, v = (rng.normal(size=(B, nch * Lc, H, D)) for _ in range(3))
    o, lse = A.block_causal_attention(q, k, v, Lc, W, 0.5)
    for b in range(B):
        for h in range(H):
            for c in range(nch):
                r = slice(c * Lc, (c + 1) * Lc)
                kr = slice(max(0, c - W) * Lc, (c + 1) * Lc)
                so, sl = _sdpa(q[b, r, h], k[b, kr, h], v[b, kr, h], 0.5)
                np.testing.assert_allclose(o[b, h, r], so, atol=1e-12)
                np.testing.assert_allclose(lse[b, h, r], sl, atol=1e-12)


def test_block_causal_row_subset_and_streaming_agree():
    """Rows of chunk c of the full-sequence pass equal streaming attention for
    chunk c with a ring holding the W previous chunks."""
    rng = np.random.default_rng(31)
    B, nch, Lc, H, D, W = 1, 6, 4, 2, 8, 2
    q, k, v = (rng.normal(size=(B, nch * Lc, H, D)) for _ in range(3))
    rows = np.array([0, 5, 9, 13, 22, 23])
    o_sub, l_sub = A.block_causal_attention(q, k, v, Lc, W, 0.4, rows=rows)
    o_all, l_all = A.block_causal_attention(q, k, v, Lc, W, 0.4)
    np.testing.assert_allclose(o_sub, o_all[:, :, rows], atol=1e-14)
    ring = ListRing(W)
    qb, kb, vb = (_blhd_to_bhld(x) for x in (q, k, v))
    for c in range(nch):
        sl = slice(c * Lc, (c + 1) * Lc)
        o, l = A.streaming_chunk_attention(qb[:, :, sl], ring, c, kb[:, :, sl], vb[:, :, sl], W, False, 0.4)
        np.testing.assert_allclose(o, o_all[:, :, sl], atol=1e-12)
        np.testing.assert_allclose(l, l_all[:, :, sl], atol=1e-12)
        ring.append(c, kb[:, :, sl], vb[:, :, sl])


def test_block_causal_restricted_keys_equal_full_mask():
    """Leaving out the keys that no selected row can see (restrict_keys)
    gives the full-mask result: the left-out terms are exact zeros."""
    rng = np.random.default_rng(32)
    B, nch, Lc, H, D, W = 2, 7, 5, 2, 8, 2
    q, k, v = (rng.normal(size=(B, nch * Lc, H, D)) for _ in range(3))
    rows = np.array([0, 3, 7, 11, 12, 18, 24, 30, 34, 2, 33])  # unsorted, several per chunk
    o_r, l_r = A.block_causal_attention(q, k, v, Lc, W, 0.45, rows=rows)
    o_f, l_f = A.block_causal_attention(q, k, v, Lc, W, 0.45, rows=rows, restrict_keys=False)
    np.testing.assert_allclose(o_r, o_f, atol=1e-13)
    np.testing.assert_allclose(l_r, l_f, atol=1e-13)
    # and each row against the scalar-loop brute force over all keys
    mask_all = A.chunk_visibility(rows // Lc, np.arange(nch * Lc) // Lc, W)
    for b in range(B):
        for h in range(H):
            ob, lb = _brute(q[b, rows, h], k[b, :, h], v[b, :, h], mask_all, 0.45)
            np.testing.assert_allclose(o_r[b, h], ob, atol=1e-12)
            np.testing.assert_allclose(l_r[b, h], lb, atol=1e-12)
