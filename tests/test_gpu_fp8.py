"""GPU parity of the FP8-E4M3 KV cache: append (codes and scales bit-exact
against the oracle's quantiser) and attention over the quantised ring.

Attention is compared with the oracle run on the dequantised cache
(x_hat = E4M3 value * scale, in fp64): max-abs 5e-2 plus half a bf16 ulp of
the reference value (2^-8 relative: outlier rows reach |O| > 16, where the
single rounding of the fp32 result to bf16 alone may move it by up to 2^-8
|O| = 0.0625), and mean-abs 2e-3.
Against the un-quantised inputs the quantisation itself moves the outputs of
these outlier-heavy inputs by up to ~1 (mean ~9e-3; measured with the oracle
alone), so that comparison is checked only in the mean: the kernel may not
add more than the quantisation does."""

import numpy as np
import pytest
import torch

from oracle import fp8 as OF
from streaming_attention_block_gb300 import KVRing, SabError, synth
import streaming_attention_block_gb300 as sab

from tests._common import FP8_LSE, FP8_MAX, compare, f32, run_stream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


def _ring(w, layers=1):
    return KVRing(layers, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=sab.KV_FP8_E4M3)


# block sizes for every launch form of the 8-bit append: a cluster of CTAs
# per (tensor, b, h) block holding 2, 4, 8 or 16 vectors a thread, and one CTA
# per block (two passes) beyond that
@pytest.mark.parametrize("B,H,D,Lc,R,sink,outliers", [(1, 2, 128, 32, 2, False, False), (2, 3, 128, 200, 3, True, True),
                                                      (1, 4, 64, 405, 4, True, True), (1, 3, 128, 405, 2, True, True),
                                                      (1, 1, 128, 700, 2, False, True), (1, 2, 128, 1536, 2, False, True),
                                                      (1, 1, 128, 4160, 2, False, False)])
def test_append_fp8_bit_exact(B, H, D, Lc, R, sink, outliers):
    w = synth.Workload("t", B=B, H=H, D=D, Lc=Lc, R=R, W=1, sink=sink, outliers=outliers, kv_fp8=True, seed=9)
    ring = _ring(w)
    gen = synth.generator(9)
    base = int(sink)
    if sink:
        sk, sv = synth.sink_kv(w, gen)
        ring.set_sink(0, sk.cuda(), sv.cuda())
    hist = {}
    for c in range(2 * R + 1):
        _, k, v = synth.chunk_qkv(w, gen)
        if c == 3:
            k = torch.zeros_like(k)  # an all-zero block: scale 1, codes 0
        ring.append(0, c, k.cuda(), v.cuda())
        hist[c] = (k, v)
    torch.cuda.synchronize()
    K, V, KS, VS = (x.cpu().numpy() for x in ring.layer_views(0))
    for c in range(R + 1, 2 * R + 1):
        slot = c % R
        for which, (x, got, gs) in enumerate(((hist[c][0], K, KS), (hist[c][1], V, VS))):
            codes, scales = OF.quantize_chunk_bhld(f32(x))
            seg = got[:, :, (base + slot) * Lc:(base + slot + 1) * Lc]
            assert np.array_equal(scales, gs[:, :, base + slot]), f"scales chunk {c} tensor {which}"
            mism = np.argwhere(seg != codes)
            assert mism.size == 0, f"chunk {c} tensor {which}: {len(mism)} code mismatches, first {mism[:3]}"
    if sink:
        codes, scales = OF.quantize_chunk_bhld(f32(sk))
        assert np.array_equal(K[:, :, :Lc], codes) and np.array_equal(KS[:, :, 0], scales)


def _e4m3_tie_values():
    """Every midpoint between adjacent positive E4M3 values, its bf16
    neighbours on both sides, both signs, and 448 (so the block's absmax scale
    is exactly 1 and the device rounding decides every tie and near-tie)."""
    pos = np.unique(np.abs(OF.e4m3_decode(np.arange(0, 127, dtype=np.uint8))))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # 4 significant bits: exact in bf16
    bits = (mids.view(np.uint32) >> 16).astype(np.uint32)
    near = np.concatenate([bits, bits + 1, bits - 1]) << 16  # bf16 neighbours (positive values)
    vals = near.astype(np.uint32).view(np.float32)
    vals = np.concatenate([vals, -vals, [448.0, -448.0]]).astype(np.float32)
    assert np.max(np.abs(vals)) == 448.0
    return vals


def test_append_fp8_device_rounding_at_ties():
    """The device conversion against the oracle codec on every E4M3 midpoint
    and its bf16 neighbours (scale fixed at 1 by a 448 in the block)."""
    vals = _e4m3_tie_values()
    Lc, D = 128, 128
    x = np.zeros(Lc * D, dtype=np.float32)
    x[:len(vals)] = vals
    x = torch.from_numpy(x.reshape(1, Lc, 1, D)).to(torch.bfloat16)
    assert np.array_equal(x.float().numpy().reshape(-1)[:len(vals)], vals)  # all exact in bf16
    w = synth.Workload("ties", B=1, H=1, D=D, Lc=Lc, R=2, W=1, kv_fp8=True, seed=1)
    ring = _ring(w)
    ring.append(0, 0, x.cuda(), (-x).cuda())
    torch.cuda.synchronize()
    K, V, KS, VS = (t.cpu().numpy() for t in ring.layer_views(0))
    for got, gs, src in ((K, KS, x), (V, VS, -x)):
        codes, scales = OF.quantize_chunk_bhld(f32(src))
        assert scales[0, 0] == 1.0 and gs[0, 0, 0] == 1.0
        mism = np.argwhere(got[:, :, :Lc] != codes)
        assert mism.size == 0, f"{len(mism)} code mismatches at ties, first {mism[:3]}"


SMALL = [
    ("fp8_small", synth.Workload("f8", B=1, H=2, D=128, Lc=200, R=3, W=2, chunks=7, sink=True, kcur_separate=False,
                                 kv_fp8=True, outliers=True, seed=51), 1),
    ("fp8_small_split3", synth.Workload("f8", B=2, H=2, D=128, Lc=160, R=4, W=3, chunks=9, sink=True,
                                        kcur_separate=False, kv_fp8=True, outliers=True, seed=52), 3),
]


def _fp8(O, L, o_ref, l_ref, rows=None, what=""):
    return compare(O, L, o_ref, l_ref, rows=rows, max_tol=FP8_MAX, mean_tol=2e-3, lse_tol=FP8_LSE, what=what,
                   rel_ulp=2.0 ** -8)


def _raw(O, L, o_ref, l_ref, rows=None, what=""):
    return compare(O, L, o_ref, l_ref, rows=rows, max_tol=np.inf, mean_tol=2e-2, lse_tol=np.inf, what=what)


@pytest.mark.parametrize("name,w,splits", SMALL, ids=[s[0] for s in SMALL])
def test_fp8_attention_small(name, w, splits):
    ring = _ring(w)
    res, _ = run_stream(w, ring, check_chunks=set(range(w.chunks)), splits=splits, on_check=_fp8)
    assert len(res) == w.chunks
    ring2 = _ring(w)
    run_stream(w, ring2, check_chunks=set(range(w.chunks)), splits=splits, on_check=_raw, fp8_reference="raw")
    assert sab.get_last_device_error() == 0


def test_fp8_long_window_sampled_rows():
    """FP8 cache at the sink + 20-slot ring shape, 60 chunks, 8 KV splits;
    checked on both sides of every wrap ({0, 1, 18, 19, 20, 21, 39, 40, 59})."""
    w = synth.workload("fp8_kv")
    rows = np.concatenate([np.arange(0, 405, 9), [404]])
    ring = _ring(w)
    res, _ = run_stream(w, ring, check_chunks={0, 1, 18, 19, 20, 21, 39, 40, 59}, rows=rows, on_check=_fp8)
    assert len(res) == 9
    assert sab.get_last_device_error() == 0


def test_fp8_long_window_auto_sampled_rows():
    """The same stream through the library's own launch choice
    (num_splits = 0, as the benchmark times it) on both sides of every wrap."""
    w = synth.workload("fp8_kv")
    rows = np.concatenate([np.arange(0, 405, 7), [404]])
    res, _ = run_stream(w, _ring(w), check_chunks={0, 1, 18, 19, 20, 21, 39, 40, 59}, rows=rows, splits=0, on_check=_fp8)
    assert len(res) == 9
    assert sab.get_last_device_error() == 0


def test_fp8_unsupported_forms():
    w = synth.Workload("u", B=1, H=2, D=128, Lc=64, R=2, W=1, kv_fp8=True, seed=3)
    ring = _ring(w)
    q, k, v = (x.cuda() for x in synth.chunk_qkv(w, synth.generator(3)))
    ring.append(0, 0, k, v)
    with pytest.raises(SabError) as e:
        ring.attention(0, 1, q, k, v, window=1)  # current chunk passed in: not on the FP8 path
    assert e.value.status == 2
    w64 = synth.Workload("u", B=1, H=2, D=64, Lc=128, R=2, W=1, kv_fp8=True, seed=3)
    r64 = _ring(w64)
    q6, k6, v6 = (x.cuda() for x in synth.chunk_qkv(w64, synth.generator(3)))
    r64.append(0, 0, k6, v6)
    with pytest.raises(SabError) as e:
        r64.attention(0, 0, q6, window=1)  # head_dim 64
    assert e.value.status == 2
    ws = synth.Workload("u", B=1, H=2, D=128, Lc=96, R=2, W=1, kv_fp8=True, seed=3)
    rs = _ring(ws)
    qs, ks, vs = (x.cuda() for x in synth.chunk_qkv(ws, synth.generator(3)))
    rs.append(0, 0, ks, vs)
    with pytest.raises(SabError) as e:
        rs.attention(0, 0, qs, window=1)  # chunks shorter than a key tile
    assert e.value.status == 2
    torch.cuda.synchronize()
