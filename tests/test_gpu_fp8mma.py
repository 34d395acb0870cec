"""GPU parity of chunk attention with E4M3 tensor-core products
(``sab_chunk_attention_fp8mma``) against the oracle of ``oracle/fp8mma.py``.

The oracle quantises each query row exactly as the kernel does (the same
fp32 decisions), uses the cache's dequantised keys and values, and returns
the exact result with a per-element bound on what rounding P to E4M3 can
change.  Tolerance per element: that bound, plus one bf16 ulp of the result
(2^-8 |O|) and 1e-3 for the fp32 accumulations and the approximate
exponential; LSE within 2e-3 (P is not rounded in the row sums, so LSE only
sees the fp32 score accumulation of exact E4M3 products).  The bulk is held
to the oracle's statistical model of the rounding: over each checked call,
mean |error| <= 1.25 x mean(sqrt(2/pi) sigma) + 2^-10 mean |O| + 1e-4, with
sigma the standard deviation of uniform rounding of every P to E4M3 and the
second term the bf16 rounding of the output.  The kernel's mean error is
0.88-0.99 of the model's on these workloads; a P rounding toward zero
instead of to nearest lands at 1.22-1.32 of the limit
(``tests/test_oracle_fp8mma.py::test_mean_check_rejects_truncated_p``)."""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import fp8 as O8
from oracle import fp8mma as OF
from oracle.ring import ListRing
from streaming_attention_block_gb300 import synth
import streaming_attention_block_gb300 as sab

from ._common import bhld, f64

pytestmark = pytest.mark.gpu

MEAN_FACTOR = 1.25  # mean error allowed, in units of the uniform-rounding model's mean


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


def _quantised(x_blhd):
    codes, scales = O8.quantize_chunk_bhld(x_blhd.float().numpy())
    deq = np.empty(codes.shape, dtype=np.float64)
    for b in range(codes.shape[0]):
        for h in range(codes.shape[1]):
            deq[b, h] = O8.dequantize_block(codes[b, h], scales[b, h])
    return deq, scales


def _stream(w, check_chunks, rows=None, splits=1):
    """Append-first stream over an E4M3 ring (``splits`` KV partitions, 0 =
    the library's choice); at ``check_chunks`` compare every (b, h) on
    ``rows``.  Returns the worst error / tolerance ratio and, per
    checked chunk, the mean error and the predicted mean rounding error."""
    gen = synth.generator(w.seed)
    ring = sab.KVRing(1, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=sab.KV_FP8_E4M3)
    oring = ListRing(w.R)
    vscale = {}  # chunk id -> V scales [B, H]
    if w.sink:
        sk, sv = synth.sink_kv(w, gen)
        ring.set_sink(0, sk.cuda(), sv.cuda())
        (kq, _), (vq, vsc) = _quantised(sk), _quantised(sv)
        oring.set_sink(kq, vq)
        vscale[OA.SINK_CHUNK] = vsc
    worst, stats = 0.0, []
    ws = ring.workspace(splits) if splits != 1 else None
    rsel = slice(None) if rows is None else rows
    for c in range(w.chunks):
        q, k, v = synth.chunk_qkv(w, gen)
        ring.append(0, c, k.cuda(), v.cuda())
        (kq, _), (vq, vsc) = _quantised(k), _quantised(v)
        oring.append(c, kq, vq)
        vscale[c] = vsc
        O = torch.empty((w.B, w.Lc, w.H, w.D), dtype=torch.bfloat16, device="cuda")
        LSE = torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda")
        sab.chunk_attention_fp8mma(ring.handle, 0, c, q.cuda(), w.W, w.sink, w.scale, O, LSE, num_splits=splits,
                                   workspace=ws)
        if c not in check_chunks:
            continue
        torch.cuda.synchronize()
        assert sab.get_last_device_error() == 0
        K, V, kid, ksink = OA.streaming_key_set(oring, c, None, None, w.W, w.sink)
        qq = bhld(q)[:, :, rsel]
        mask = OA.chunk_visibility(np.full(qq.shape[2], c), kid, w.W, ksink)
        o_gpu = bhld(O)[:, :, rsel]
        l_gpu = f64(LSE)[:, :, rsel]
        e_sum = p_sum = o_sum = 0.0
        for b in range(w.B):
            for h in range(w.H):
                vs_key = np.array([vscale[int(i)][b, h] for i in kid], dtype=np.float64)
                o, lse, bound = OF.head_attention(qq[b, h].astype(np.float32), K[b, h], V[b, h], mask, w.scale,
                                                  vs_key)
                err = np.abs(o_gpu[b, h] - o)
                tol = bound + 2.0 ** -8 * np.abs(o) + 1e-3
                worst = max(worst, float(np.max(err / tol)))
                sigma = OF.rounding_sigma(qq[b, h].astype(np.float32), K[b, h], V[b, h], mask, w.scale, vs_key)
                e_sum += float(np.mean(err))
                p_sum += float(np.mean(np.sqrt(2.0 / np.pi) * sigma))
                o_sum += float(np.mean(np.abs(o)))
                assert np.all(err <= tol), (f"chunk {c} b{b} h{h}: max err {err.max():.3e}, worst ratio "
                                            f"{np.max(err / tol):.2f}")
                assert np.max(np.abs(l_gpu[b, h] - lse)) <= 2e-3, f"chunk {c} b{b} h{h}: LSE"
        n = w.B * w.H
        stats.append((c, e_sum / n, p_sum / n))
        assert e_sum <= MEAN_FACTOR * p_sum + 2.0 ** -10 * o_sum + 1e-4 * n, (c, e_sum / n, p_sum / n)
    return worst, stats


@pytest.mark.parametrize("splits", [1, 3, 0], ids=["unsplit", "3splits", "auto"])
def test_fp8mma_small_elementwise(splits):
    """Sink + 3-slot ring, 200-token chunks (key tiles straddle chunks),
    window 2, 1% x8 outliers; every row of chunks 0, 1, 3 and 5, unsplit, in
    three KV partitions merged by log-sum-exp, and with the library's split
    choice."""
    w = synth.Workload("f8s", B=1, H=2, D=128, Lc=200, R=3, W=2, chunks=6, sink=True, kcur_separate=False,
                       kv_fp8=True, outliers=True, seed=41)
    _stream(w, {0, 1, 3, 5}, splits=splits)


@pytest.mark.parametrize("splits", [1, 0], ids=["unsplit", "auto"])
def test_fp8mma_full_size_sampled_rows(splits):
    """Long-window FP8 workload (H24, 405-token chunks, sink + 20-slot ring,
    window 19, 60 chunks so the ring wraps 3 times): sampled rows of the
    chunks on both sides of every wrap, every head; unsplit and with the
    library's split choice (the launch the benchmark times)."""
    w = synth.workload("fp8_kv")
    rows = np.concatenate([np.arange(0, w.Lc, 9), [w.Lc - 1]])
    _stream(w, {0, 1, 18, 19, 20, 21, 39, 40, 59}, rows=rows, splits=splits)


def test_fp8mma_argument_errors():
    """Host-side refusals of the E4M3-product entry: a bf16 ring is
    UNSUPPORTED, a split call without a workspace (explicit splits, or the
    library's choice when it picks more than one) is WORKSPACE, a workspace
    sized for fewer splits is WORKSPACE, a split count past the limit is
    INVALID_ARG; nothing is launched for any of them."""
    w = synth.Workload("f8e", B=1, H=2, D=128, Lc=256, R=3, W=2, kv_fp8=True, seed=43)
    ring = sab.KVRing(1, w.B, w.H, w.D, w.Lc, w.R, kv_dtype=sab.KV_FP8_E4M3)
    gen = synth.generator(w.seed)
    for c in range(3):
        q, k, v = synth.chunk_qkv(w, gen)
        ring.append(0, c, k.cuda(), v.cuda())
    qd = q.cuda()
    O = torch.full_like(qd, 7.0)
    LSE = torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda")
    with pytest.raises(sab.SabError) as e:
        sab.chunk_attention_fp8mma(ring.handle, 0, 2, qd, w.W, False, w.scale, O, LSE, num_splits=3)
    assert e.value.status == 4  # SAB_ERR_WORKSPACE
    small = ring.workspace(2)
    with pytest.raises(sab.SabError) as e:
        sab.chunk_attention_fp8mma(ring.handle, 0, 2, qd, w.W, False, w.scale, O, LSE, num_splits=3, workspace=small)
    assert e.value.status == 4
    with pytest.raises(sab.SabError) as e:
        sab.chunk_attention_fp8mma(ring.handle, 0, 2, qd, w.W, False, w.scale, O, LSE, num_splits=1 << 20)
    assert e.value.status == 1  # SAB_ERR_INVALID_ARG
    bring = sab.KVRing(1, w.B, w.H, w.D, w.Lc, w.R)
    with pytest.raises(sab.SabError) as e:
        sab.chunk_attention_fp8mma(bring.handle, 0, 0, qd, w.W, False, w.scale, O, LSE)
    assert e.value.status == 2  # SAB_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((O == 7.0).all())
    assert sab.get_last_device_error() == 0
