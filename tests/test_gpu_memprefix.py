"""GPU parity of block-causal attention behind a variable-length memory
prefix (forward and gradients) against the fp64 oracle
(``oracle/memprefix.py``), through the C-ABI.

Forward: the bf16 bounds of the block-causal tests on every real row; padded
rows must be exactly O = 0, LSE = -inf.  Gradients: the per-element error
scale of the gradient oracle, as in the block-causal backward tests, and
exact zeros at padded positions."""

import numpy as np
import pytest
import torch

from oracle import memprefix as OM
from streaming_attention_block_gb300 import synth
import streaming_attention_block_gb300 as sab

from ._common import compare, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


CASES = [
    # name, B, H, D, Lc, W, target chunks, mem_pad, mem_lens
    ("tile_memory", 2, 2, 128, 128, 1, 3, 200, (200, 77)),
    ("ragged_d64", 2, 2, 64, 100, 2, 4, 45, (0, 45)),
    ("long_memory", 2, 1, 128, 64, 1, 5, 300, (129, 300)),
    ("no_targets_left", 1, 2, 128, 96, 0, 2, 130, (1,)),
]


def _run(B, H, D, Lc, W, n_chunks, M, lens, seed, backward=True):
    w = synth.Workload("mp", B=B, H=H, D=D, Lc=Lc, W=W, seq_chunks=n_chunks, mem_pad=M, mem_lens=lens, seed=seed)
    gen = synth.generator(seed)
    q, k, v = synth.full_sequence_qkv(w, gen)
    do = synth.randn_bf16(gen, tuple(q.shape), "cpu")
    L = q.shape[1]
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    ml = torch.tensor(lens, dtype=torch.int32, device="cuda")
    O = torch.empty_like(qd)
    LSE = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    sab.memory_prefix_attention(qd, kd, vd, M, ml, Lc, W, D ** -0.5, O, LSE)
    grads = None
    if backward:
        grads = tuple(torch.empty_like(qd) for _ in range(3))
        sab.memory_prefix_attention_backward(qd, kd, vd, O, dod, LSE, M, ml, Lc, W, D ** -0.5, *grads)
    torch.cuda.synchronize()
    assert sab.get_last_device_error() == 0
    return (q, k, v, do), O, LSE, grads


def _check_forward(O, LSE, o_ref, l_ref, M, lens, rows, what):
    for b, P in enumerate(lens):
        real = np.array([r for r in rows if r < P or r >= M], dtype=np.int64)
        pad = np.array([i for i, r in enumerate(rows) if P <= r < M], dtype=np.int64)
        sel = np.searchsorted(rows, real)
        if real.size:
            compare(O[b:b + 1], LSE[b:b + 1], o_ref[b:b + 1][:, :, sel], l_ref[b:b + 1][:, :, sel], rows=real,
                    what=f"{what} b{b}")
        if pad.size:
            o = O[b][torch.as_tensor(rows[pad])].float()
            assert torch.all(o == 0), f"{what} b{b}: padded rows not zero"
            assert torch.all(torch.isneginf(LSE[b][:, torch.as_tensor(rows[pad])])), f"{what} b{b}: LSE of padding"


@pytest.mark.parametrize("name,B,H,D,Lc,W,n,M,lens", CASES, ids=[c[0] for c in CASES])
def test_memory_prefix_elementwise(name, B, H, D, Lc, W, n, M, lens):
    (q, k, v, do), O, LSE, grads = _run(B, H, D, Lc, W, n, M, lens, seed=31 + M)
    L = q.shape[1]
    scale = D ** -0.5
    o_ref, l_ref = OM.memory_prefix_attention(f64(q), f64(k), f64(v), M, lens, Lc, W, scale)
    _check_forward(O, LSE, o_ref, l_ref, M, lens, np.arange(L), name)
    refs, bounds = OM.memory_prefix_attention_backward(f64(q), f64(k), f64(v), f64(do), M, lens, Lc, W, scale)
    for nm, got, ref, bnd in zip(("dQ", "dK", "dV"), grads, refs, bounds):
        g = f64(got.cpu())
        err = np.abs(g - ref)
        tol = 2.0 ** -6 * bnd + 2.0 ** -8 * np.abs(ref) + 1e-5
        bad = np.argwhere(err > tol)
        assert bad.size == 0, (f"{name} {nm}: {len(bad)} elements out of tolerance; max err {err.max():.3e}, "
                               f"worst ratio {np.max(err / tol):.2f}, first {bad[:3]}")
        for b, P in enumerate(lens):
            assert np.all(g[b, P:M] == 0.0), f"{name} {nm}: gradient at padded positions"


def test_memory_prefix_training_shape_sampled_rows():
    """Compressed-memory training shape: B2, H12, D128, 4 target chunks of
    1536 behind 3072 memory positions (one sample full, one with 1900 real),
    window 3: forward rows sampled in the memory, the padding and every chunk,
    against the oracle; gradients are finite and zero on the padding."""
    w = synth.workload("memory_prefix")
    (q, k, v, do), O, LSE, grads = _run(w.B, w.H, w.D, w.Lc, w.W, w.seq_chunks, w.mem_pad, w.mem_lens, w.seed)
    L = q.shape[1]
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 1899, 1900, 3071, 3072, 4607, 4608, L - 1], rng.integers(0, L, 20)]))
    o_ref, l_ref = OM.memory_prefix_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.mem_pad,
                                              w.mem_lens, w.Lc, w.W, w.scale, rows=rows)
    _check_forward(O, LSE, o_ref, l_ref, w.mem_pad, w.mem_lens, rows, "memory prefix, training shape")
    for g in grads:
        assert bool(torch.isfinite(g.float()).all())
        assert bool((g[1, w.mem_lens[1]:w.mem_pad].float() == 0).all())
