"""GPU parity of the INT8-key / FP8-value cache ("Matrix-Game 4.0", section
"技术新颖性": each window interval caches INT8 keys and FP8 values): append
(INT8 key codes, E4M3 value codes and both scales bit-exact against the
oracle's quantisers) and attention over the quantised ring, unsplit and split.

Attention is compared with the oracle on the dequantised cache
(x_hat = code * scale, fp64) at the FP8 tolerances (the kernel expands the
codes exactly and applies the scales in fp32), and with the un-quantised
inputs in the mean only (the quantisation itself moves the outputs)."""

import numpy as np
import pytest
import torch

from oracle import fp8 as OF
from oracle import int8 as OI
from streaming_attention_block_gb300 import KVRing, synth
import streaming_attention_block_gb300 as sab

from tests._common import FP8_LSE, FP8_MAX, compare, f32, run_stream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


def _ring(w, layers=1):
    return KVRing(layers, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=sab.KV_INT8K_FP8V)


@pytest.mark.parametrize("B,H,D,Lc,R,sink", [(1, 2, 128, 32, 2, False), (2, 3, 128, 200, 3, True),
                                             (1, 4, 64, 405, 4, True), (1, 2, 128, 1536, 2, False),
                                             (1, 1, 128, 4160, 2, False)])
def test_append_int8k_bit_exact(B, H, D, Lc, R, sink):
    w = synth.Workload("t", B=B, H=H, D=D, Lc=Lc, R=R, W=1, sink=sink, outliers=True, kv_fp8=True, kv_int8k=True,
                       seed=19)
    ring = _ring(w)
    gen = synth.generator(19)
    base = int(sink)
    if sink:
        sk, sv = synth.sink_kv(w, gen)
        ring.set_sink(0, sk.cuda(), sv.cuda())
    hist = {}
    for c in range(2 * R + 1):
        _, k, v = synth.chunk_qkv(w, gen)
        if c == 3:
            k = torch.zeros_like(k)  # an all-zero key block: scale 1, codes 0
        ring.append(0, c, k.cuda(), v.cuda())
        hist[c] = (k, v)
    torch.cuda.synchronize()
    K, V, KS, VS = (x.cpu().numpy() for x in ring.layer_views(0))
    Ki = K.view(np.int8)
    for c in range(R + 1, 2 * R + 1):
        slot = c % R
        rows = slice((base + slot) * Lc, (base + slot + 1) * Lc)
        kc, ks = OI.quantize_chunk_bhld(f32(hist[c][0]))
        vc, vs = OF.quantize_chunk_bhld(f32(hist[c][1]))
        assert np.array_equal(ks, KS[:, :, base + slot]), f"K scales chunk {c}"
        assert np.array_equal(vs, VS[:, :, base + slot]), f"V scales chunk {c}"
        mk = np.argwhere(Ki[:, :, rows] != kc)
        assert mk.size == 0, f"chunk {c}: {len(mk)} key code mismatches, first {mk[:3]}"
        mv = np.argwhere(V[:, :, rows] != vc)
        assert mv.size == 0, f"chunk {c}: {len(mv)} value code mismatches, first {mv[:3]}"
    assert Ki.min() >= -127  # the symmetric range never produces -128
    if sink:
        kc, ks = OI.quantize_chunk_bhld(f32(sk))
        assert np.array_equal(Ki[:, :, :Lc], kc) and np.array_equal(KS[:, :, 0], ks)


CASES = [
    ("int8k_small", synth.Workload("i8", B=1, H=2, D=128, Lc=200, R=3, W=2, chunks=7, sink=True, kcur_separate=False,
                                   kv_fp8=True, kv_int8k=True, outliers=True, seed=61), 1),
    ("int8k_small_split3", synth.Workload("i8", B=2, H=2, D=128, Lc=160, R=4, W=3, chunks=9, sink=True,
                                          kcur_separate=False, kv_fp8=True, kv_int8k=True, outliers=True, seed=62), 3),
]


def _deq(O, L, o_ref, l_ref, rows=None, what=""):
    return compare(O, L, o_ref, l_ref, rows=rows, max_tol=FP8_MAX, mean_tol=2e-3, lse_tol=FP8_LSE, what=what,
                   rel_ulp=2.0 ** -8)


def _raw(O, L, o_ref, l_ref, rows=None, what=""):
    return compare(O, L, o_ref, l_ref, rows=rows, max_tol=np.inf, mean_tol=2e-2, lse_tol=np.inf, what=what)


@pytest.mark.parametrize("name,w,splits", CASES, ids=[c[0] for c in CASES])
def test_int8k_attention_small(name, w, splits):
    res, _ = run_stream(w, _ring(w), check_chunks=set(range(w.chunks)), splits=splits, on_check=_deq)
    assert len(res) == w.chunks
    run_stream(w, _ring(w), check_chunks=set(range(w.chunks)), splits=splits, on_check=_raw, fp8_reference="raw")
    assert sab.get_last_device_error() == 0


def test_int8k_long_window_sampled_rows():
    """INT8-key cache at the sink + 20-slot ring shape, 60 chunks, library's
    launch choice (as the benchmark times it), on both sides of every wrap."""
    w = synth.workload("int8k_kv")
    rows = np.concatenate([np.arange(0, 405, 7), [404]])
    res, _ = run_stream(w, _ring(w), check_chunks={0, 1, 18, 19, 20, 21, 39, 40, 59}, rows=rows, splits=0, on_check=_deq)
    assert len(res) == 9
    assert sab.get_last_device_error() == 0
