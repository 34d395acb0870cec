"""Pins of the E4M3-product attention oracle (``oracle/fp8mma.py``): the
per-row Q quantiser against torch's float8_e4m3fn rounding, the exact part
against the plain attention oracle on the same quantised operands, and the
P-rounding bound against a brute-force replay of the rounding (torch's E4M3
cast, running-max offsets, relative V scales down to 1/40), which a bound
that forgot the V-scale factor fails."""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import fp8mma as OF


def _e4m3_round(x):
    """Round float32 values to E4M3 with torch (independent of oracle.fp8)."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_row_quantiser_matches_torch_cast():
    rng = np.random.default_rng(1)
    q = (rng.standard_normal((64, 128)) * rng.uniform(0.01, 30, (64, 1))).astype(np.float32)
    q[3] = 0.0
    q_hat, sc = OF.quantize_rows(q)
    for i in range(q.shape[0]):
        amax = np.float32(np.max(np.abs(q[i])))
        s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
        assert sc[i] == s
        ref = _e4m3_round((q[i] / s).astype(np.float32)) * np.float64(s)
        np.testing.assert_array_equal(q_hat[i], ref)
    # every row's largest magnitude lands on the top code 448
    big = np.argmax(np.abs(q[0]))
    assert abs(q_hat[0, big]) == 448.0 * np.float64(sc[0])


def test_exact_part_is_plain_attention_on_quantised_operands():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((40, 32)).astype(np.float32)
    k, v = rng.standard_normal((2, 90, 32))
    mask = rng.random((40, 90)) < 0.6
    mask[:, 0] = True
    o, lse, _ = OF.head_attention(q, k, v, mask, 0.2, np.ones(90))
    q_hat, _ = OF.quantize_rows(q)
    o2, l2 = OA.masked_attention(q_hat, k, v, mask, 0.2)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, l2, rtol=0, atol=1e-13)


def _replay(q, k, v, mask, scale, vs, delta, bound_fn=None, gain=OF.P_GAIN_LOG2):
    """Round P the way the product sees it: P * r * 2^(gain + delta) to E4M3
    and back."""
    o, lse, bound = OF.head_attention(q, k, v, mask, scale, vs, gain)
    q_hat, _ = OF.quantize_rows(q)
    s = np.where(mask, scale * (q_hat @ k.T), -np.inf)
    p = np.where(mask, np.exp(s - s.max(axis=1, keepdims=True)), 0.0)
    vs_ref = vs[mask.any(axis=0)].max()
    r = vs / vs_ref
    f = r[None, :] * 2.0 ** (gain + delta)
    assert np.all(p * f <= 448.0)
    p_q = _e4m3_round(p * f) / f
    o_sim = (p_q @ v) / p.sum(axis=1, keepdims=True)
    if bound_fn is not None:
        e = np.where(mask, bound_fn(p, r), 0.0)
        bound = (e @ np.abs(v)) / p.sum(axis=1, keepdims=True)
    return np.abs(o_sim - o), bound


@pytest.mark.parametrize("peak", [0.3, 3.0, 12.0])
@pytest.mark.parametrize("delta", [0, 2, 4])
def test_bound_holds_under_brute_force_rounding(peak, delta):
    rng = np.random.default_rng(int(peak * 10) + delta)
    Nk, D = 600, 64
    q = (rng.standard_normal((48, D)) * peak).astype(np.float32)
    k = rng.standard_normal((Nk, D))
    v = rng.standard_normal((Nk, D))
    # three chunks with very different V scales; one with 8x outliers
    vs = np.repeat([0.05, 0.9, 2.0], Nk // 3)
    v[400:] *= 1.0
    v[rng.random((Nk, D)) < 0.01] *= 8.0
    mask = np.ones((48, Nk), dtype=bool)
    mask[::3, 450:] = False
    err, bound = _replay(q, k, v, mask, 1.0 / np.sqrt(D), vs, delta)
    assert np.all(err <= bound + 1e-12), float(np.max(err - bound))
    assert np.mean(bound) < 2.0 ** -3 * np.mean(np.abs(v))  # not vacuous (the leading term is 2^-4)


def test_bound_without_the_scale_factor_fails():
    """One dominant key (r = 1) and 390 keys of equal score whose V scale is
    1/40 of it, with no gain: P r = 1.49 * 2^-9 rounds down by 0.49 subnormal
    steps for all of them at once (coherent error).  The bound holds; a bound
    that forgot the relative V scale r is violated."""
    D, Nk = 32, 400
    p0 = 1.49 * 2.0 ** -9 * 40.0
    q = np.zeros((4, D), dtype=np.float32)
    q[:, 0] = 1.0
    k = np.zeros((Nk, D))
    k[0, 0] = 2.0
    k[1:391, 0] = 2.0 + np.log(p0)
    k[391:, 0] = -3.0
    v = np.ones((Nk, D))
    vs = np.ones(Nk)
    vs[1:391] = 0.025
    mask = np.ones((4, Nk), dtype=bool)
    wrong = lambda p, r: np.where(p >= 2.0 ** -6, 2.0 ** -4 * p, np.minimum(p, 2.0 ** -10))
    err, bad_bound = _replay(q, k, v, mask, 1.0, vs, 0, bound_fn=wrong, gain=0)
    assert np.all(err > 4 * bad_bound)
    err, bound = _replay(q, k, v, mask, 1.0, vs, 0, gain=0)
    assert np.all(err <= bound + 1e-12)
    assert np.all(err >= 0.9 * bound)  # and it is tight here


def test_gain_shrinks_the_subnormal_term():
    """With the kernel's gain the same coherent case is 2^g times tighter and
    still covered."""
    D, Nk = 32, 400
    p0 = 1.49 * 2.0 ** -9 * 40.0 / 2.0 ** OF.P_GAIN_LOG2  # P r 2^g = 1.49 * 2^-9
    q = np.zeros((4, D), dtype=np.float32)
    q[:, 0] = 1.0
    k = np.zeros((Nk, D))
    k[0, 0] = 2.0
    k[1:391, 0] = 2.0 + np.log(p0)
    k[391:, 0] = -3.0
    v = np.ones((Nk, D))
    vs = np.ones(Nk)
    vs[1:391] = 0.025
    mask = np.ones((4, Nk), dtype=bool)
    err, bound = _replay(q, k, v, mask, 1.0, vs, 0)
    assert np.all(err <= bound + 1e-12)
    err0, bound0 = _replay(q, k, v, mask, 1.0, vs, 0, gain=0)
    assert np.all(bound < bound0)


@pytest.mark.parametrize("peak", [0.3, 3.0])
def test_sigma_predicts_the_replayed_error(peak):
    """The uniform-rounding model's sigma matches the RMS of the replayed
    rounding error (random keys: errors independent across keys)."""
    rng = np.random.default_rng(11 + int(peak))
    Nk, D = 800, 64
    q = (rng.standard_normal((64, D)) * peak).astype(np.float32)
    k = rng.standard_normal((Nk, D))
    v = rng.standard_normal((Nk, D))
    vs = np.repeat([0.3, 1.0], Nk // 2)
    mask = np.ones((64, Nk), dtype=bool)
    err, _ = _replay(q, k, v, mask, 1.0 / np.sqrt(D), vs, 0)
    sigma = OF.rounding_sigma(q, k, v, mask, 1.0 / np.sqrt(D), vs)
    ratio = np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(sigma ** 2))
    assert 0.7 < ratio < 1.3, ratio
    # and the mean magnitude is about sqrt(2/pi) sigma
    ratio_abs = np.mean(err) / np.mean(np.sqrt(2 / np.pi) * sigma)
    assert 0.7 < ratio_abs < 1.3, ratio_abs


def _e4m3_truncate(x):
    """Round positive float32 values toward zero onto the E4M3 grid (the
    grid taken from torch's float8_e4m3fn codes 0..126)."""
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = np.asarray(x, dtype=np.float64)
    return grid[np.searchsorted(grid, x, side="right") - 1]


@pytest.mark.parametrize("peak", [0.3, 3.0])
def test_mean_check_rejects_truncated_p(peak):
    """The GPU test's mean check (mean |error| <= 1.25 x mean(sqrt(2/pi) sigma)
    + 2^-10 mean |O| + 1e-4) has teeth: a P path that rounds toward zero
    instead of to nearest -- a plausible conversion bug that the per-element
    bound alone lets through -- doubles the mean-square rounding error and
    fails it, while round-to-nearest passes on the same inputs."""
    rng = np.random.default_rng(23 + int(peak))
    Nk, D = 800, 64
    q = (rng.standard_normal((64, D)) * peak).astype(np.float32)
    k = rng.standard_normal((Nk, D))
    v = rng.standard_normal((Nk, D))
    vs = np.repeat([0.3, 1.0], Nk // 2)
    mask = np.ones((64, Nk), dtype=bool)
    scale = 1.0 / np.sqrt(D)
    o, _, bound = OF.head_attention(q, k, v, mask, scale, vs)
    sigma = OF.rounding_sigma(q, k, v, mask, scale, vs)
    q_hat, _ = OF.quantize_rows(q)
    s = scale * (q_hat @ k.T)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    f = (vs / vs.max())[None, :] * 2.0 ** OF.P_GAIN_LOG2
    limit = 1.25 * np.mean(np.sqrt(2.0 / np.pi) * sigma) + 2.0 ** -10 * np.mean(np.abs(o)) + 1e-4
    for rounder, passes in ((_e4m3_round, True), (_e4m3_truncate, False)):
        o_sim = ((rounder(p * f) / f) @ v) / p.sum(axis=1, keepdims=True)
        err = np.abs(o_sim - o)
        assert np.all(err <= bound + 2.0 ** -8 * np.abs(o) + 1e-3)  # the per-element bound holds for both
        assert (np.mean(err) <= limit) == passes, (rounder.__name__, float(np.mean(err)), float(limit))
