"""GPU parity of the block-causal attention backward against the fp64
gradient oracle (``oracle/backward.py``), on the same bf16 inputs.

The GPU path runs the GPU forward for O and LSE, then the backward.  Error
budget per output element (derived from the arithmetic): P and dS are
rounded to bf16 before the gradient MMAs (2^-9 relative each), delta uses
the bf16 forward output, the MMAs accumulate exact bf16 products in fp32,
and the result is rounded to bf16 once -- so |gpu - ref| <= 2^-6 * bound +
2^-8 * |ref| + 1e-5, with the oracle's per-element error scale ``bound``
(an 8x margin over the first-order estimate 2^-9 * bound)."""

import numpy as np
import pytest
import torch

from oracle import backward as OB
from streaming_attention_block_gb300 import synth
import streaming_attention_block_gb300 as sab

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


CASES = [
    # (B, L, H, D, chunk_tokens, window)
    ("aligned", 1, 640, 2, 128, 128, 1),
    ("ragged_d64", 2, 500, 2, 64, 100, 2),
    ("long_chunks", 1, 3 * 1536, 2, 128, 1536, 2),
    ("chunk_local_w0", 1, 384, 2, 128, 128, 0),
    ("window_past_start", 1, 448, 1, 128, 64, 9),
]


@pytest.mark.parametrize("name,B,L,H,D,Lc,W", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(name, B, L, H, D, Lc, W):
    gen = torch.Generator().manual_seed(4242 + L)
    q, k, v, do = (synth.randn_bf16(gen, (B, L, H, D), "cpu") for _ in range(4))
    scale = D ** -0.5
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    O = torch.empty_like(qd)
    LSE = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    sab.block_causal_attention(qd, kd, vd, Lc, W, 1, scale, O, LSE)
    dQ, dK, dV = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    sab.block_causal_attention_backward(qd, kd, vd, O, dod, LSE, Lc, W, scale, dQ, dK, dV)
    torch.cuda.synchronize()
    assert sab.get_last_device_error() == 0
    f64 = lambda t: t.float().numpy().astype(np.float64)
    refs, bounds = OB.block_causal_attention_backward(f64(q), f64(k), f64(v), f64(do), Lc, W, scale,
                                                      abs_bounds=True)
    for nm, got, ref, bnd in zip(("dQ", "dK", "dV"), (dQ, dK, dV), refs, bounds):
        g = f64(got.cpu())
        err = np.abs(g - ref)
        tol = 2.0 ** -6 * bnd + 2.0 ** -8 * np.abs(ref) + 1e-5
        bad = np.argwhere(err > tol)
        assert bad.size == 0, (f"{name} {nm}: {len(bad)} elements out of tolerance; max err {err.max():.3e}, "
                               f"worst ratio {np.max(err / tol):.2f}, first {bad[:3]}")
        # and the bulk is far tighter than the bound
        assert np.mean(err) <= 2.0 ** -8 * np.mean(np.abs(ref)) + 1e-5, f"{name} {nm}: mean error too large"


def test_backward_full_size_sampled_rows():
    """Training shape: B2 x 30720 tokens (20 chunks of 1536), H12, D128,
    window 2, in the launch configuration the benchmark times; dQ at query
    rows and dK, dV at key rows sampled at chunk edges and inside, for a few
    (batch, head) pairs, against the row-restricted oracle."""
    w = synth.workload("block_causal")
    gen = synth.generator(w.seed)
    q, k, v = synth.full_sequence_qkv(w, gen)
    do = synth.randn_bf16(gen, tuple(q.shape), "cpu")
    L = w.seq_chunks * w.Lc
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    O = torch.empty_like(qd)
    LSE = torch.empty((w.B, w.H, L), dtype=torch.float32, device="cuda")
    sab.block_causal_attention(qd, kd, vd, w.Lc, w.W, 1, w.scale, O, LSE)
    dQ, dK, dV = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    sab.block_causal_attention_backward(qd, kd, vd, O, dod, LSE, w.Lc, w.W, w.scale, dQ, dK, dV)
    torch.cuda.synchronize()
    assert sab.get_last_device_error() == 0
    rng = np.random.default_rng(9)
    qr = np.unique(np.concatenate([[0, w.Lc - 1, w.Lc, 2 * w.Lc + 5, L - 1], rng.integers(0, L, 6)]))
    kr = np.unique(np.concatenate([[0, w.Lc - 1, 10 * w.Lc, L - w.Lc, L - 1], rng.integers(0, L, 6)]))
    f64 = lambda t: t.float().numpy().astype(np.float64)
    got = [x.cpu() for x in (dQ, dK, dV)]
    for b, h in ((0, 0), (1, 7)):
        one = [f64(x[b:b + 1, :, h:h + 1]) for x in (q, k, v, do)]
        refs, bounds = OB.block_causal_attention_backward_rows(*one, w.Lc, w.W, w.scale, 0, 0, qr, kr)
        for nm, g, rows, ref, bnd in zip(("dQ", "dK", "dV"), got, (qr, kr, kr), refs, bounds):
            err = np.abs(f64(g[b, rows, h]) - ref)
            tol = 2.0 ** -6 * bnd + 2.0 ** -8 * np.abs(ref) + 1e-5
            assert np.all(err <= tol), (f"full size {nm} (b{b} h{h}): max err {err.max():.3e}, "
                                        f"worst ratio {np.max(err / tol):.2f}")
