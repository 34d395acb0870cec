"""Pins of the QK-norm + rotary oracle (``oracle/qkrope.py``) against facts
that do not depend on it: the RMS of a normalised token is 1 (scale
invariant), rotation keeps every pair's length, position 0 is the identity,
the dot product of a rotated query and key depends only on their position
difference (the defining property of rotary embeddings), a hand-computed 2-D
rotation, and the grid coordinates of a chunk."""

import numpy as np

from oracle import qkrope as OQ


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_rms_norm_unit_rms_and_scale_invariance():
    x = _rand((2, 5, 3, 8), 1)
    y = OQ.rms_norm(x)
    rms = np.sqrt(np.mean(y.reshape(2, 5, 24) ** 2, axis=-1))
    assert np.allclose(rms, 1.0 / np.sqrt(1.0 + OQ.EPS / np.mean(x.reshape(2, 5, 24) ** 2, axis=-1)), rtol=1e-12)
    # without eps the normalisation is exactly scale invariant
    assert np.allclose(OQ.rms_norm(7.0 * x, eps=0.0), OQ.rms_norm(x, eps=0.0), rtol=1e-12)
    g = np.linspace(0.5, 2.0, 24)
    assert np.allclose(OQ.rms_norm(x, g), y * g.reshape(1, 1, 3, 8), rtol=1e-12)


def test_rotation_keeps_pair_lengths_and_position_zero_is_identity():
    x = _rand((1, 6, 2, 16), 2)
    ang = OQ.angles(OQ.positions(3, 6, (6, 1, 1)), (16, 0, 0))
    y = OQ.rope(x, ang)
    assert np.allclose(np.hypot(y[..., 0::2], y[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]), rtol=1e-12)
    ang0 = OQ.angles(OQ.positions(0, 1, (1, 1, 1)), (16, 0, 0))
    assert np.array_equal(OQ.rope(x[:, :1], ang0), x[:, :1])


def test_hand_computed_rotation():
    # D = 2, one pair, theta_0 = 1: position 2 rotates (1, 0) by 2 rad
    x = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)
    ang = OQ.angles(np.array([[2.0, 0.0, 0.0]]), (2, 0, 0))
    assert np.allclose(OQ.rope(x, ang).ravel(), [np.cos(2.0), np.sin(2.0)], rtol=0, atol=1e-15)
    # D = 4, base 10000: theta_1 = 10000^(-1/2) = 0.01
    ang4 = OQ.angles(np.array([[100.0, 0.0, 0.0]]), (4, 0, 0))
    assert np.allclose(ang4.ravel(), [100.0, 1.0], rtol=1e-12)


def test_dot_product_depends_only_on_relative_position():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 1, 12))
    k = rng.standard_normal((1, 1, 1, 12))
    bands = (4, 4, 4)

    def rot(v, p):
        return OQ.rope(v, OQ.angles(np.asarray([p], dtype=np.float64), bands))

    a = np.sum(rot(q, [5, 2, 7]) * rot(k, [3, 1, 4]))
    b = np.sum(rot(q, [12, 9, 10]) * rot(k, [10, 8, 7]))  # same (2, 1, 3) offset
    c = np.sum(rot(q, [6, 2, 7]) * rot(k, [3, 1, 4]))     # different offset
    assert np.isclose(a, b, rtol=1e-12) and not np.isclose(a, c, rtol=1e-6)


def test_grid_positions():
    p = OQ.positions(2, 12, (2, 2, 3))
    # chunk 2 of 2 frames each: frames 4, 5; rows 0..1; columns 0..2
    assert p[0].tolist() == [4, 0, 0] and p[5].tolist() == [4, 1, 2] and p[6].tolist() == [5, 0, 0]
    assert p[11].tolist() == [5, 1, 2]
