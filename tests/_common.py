"""Shared test helpers: tensor conversions and the stream driver that feeds the
same seeded inputs to the CUDA library and to the CPU oracle."""

from __future__ import annotations

import numpy as np
import torch

from oracle import attention as OA
from oracle import fp8 as OF
from oracle import int8 as OI
from oracle.ring import ListRing
from streaming_attention_block_gb300 import synth

# Tolerances fixed by the acceptance criteria of the method: BF16 outputs
# within max-abs 1e-2 and mean-abs 1e-3 of the fp64 oracle on the same
# bf16-rounded inputs; FP8-KV outputs within max-abs 5e-2.  LSE, which the
# criteria do not cover, within 1e-3 (bf16) / 5e-2 (fp8): the kernel
# accumulates the row sum in fp32 and takes one logarithm.
BF16_MAX, BF16_MEAN, BF16_LSE = 1e-2, 1e-3, 1e-3
FP8_MAX, FP8_LSE = 5e-2, 5e-2


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16/fp32 tensor -> float64 numpy (exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def f32(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> float32 numpy (exact; the oracle widens to float64 per head)."""
    return t.detach().float().cpu().numpy()


def bhld(t_blhd) -> np.ndarray:
    """token-major [B, L, H, D] -> head-major [B, H, L, D] float64."""
    x = f64(t_blhd) if isinstance(t_blhd, torch.Tensor) else np.asarray(t_blhd, dtype=np.float64)
    return np.ascontiguousarray(np.transpose(x, (0, 2, 1, 3)))


def compare(O_gpu: torch.Tensor, LSE_gpu: torch.Tensor, O_ref: np.ndarray, L_ref: np.ndarray, rows=None,
            max_tol=BF16_MAX, mean_tol=BF16_MEAN, lse_tol=BF16_LSE, what="", rel_ulp=0.0):
    """O_gpu token-major [B, L, H, D]; O_ref head-major [B, H, nrows, D] over `rows`.

    ``rel_ulp`` widens the per-element bound to max_tol + rel_ulp * |O_ref|:
    a bf16 output of magnitude >= 16 has an ulp of 0.125, so no absolute
    bound below that can hold there (used for the outlier-heavy FP8 inputs).
    """
    o = bhld(O_gpu)
    lse = f64(LSE_gpu)
    if rows is not None:
        o = o[:, :, rows]
        lse = lse[:, :, rows]
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    d = np.abs(o - O_ref)
    dl = np.abs(lse - L_ref)
    msg = f"{what}: max|dO|={d.max():.3e} mean|dO|={d.mean():.3e} max|dLSE|={dl.max():.3e}"
    assert np.all(d <= max_tol + rel_ulp * np.abs(O_ref)), msg
    if mean_tol is not None:
        assert d.mean() <= mean_tol, msg
    assert dl.max() <= lse_tol, msg
    return d.max(), d.mean(), dl.max()


def oracle_kv(k_blhd: torch.Tensor, v_blhd: torch.Tensor, fp8: bool, int8k: bool = False):
    """What the oracle caches for a chunk: bf16 values, or the dequantised codes
    of the per-(b, h) absmax quantisers (E4M3 keys, or INT8 keys with
    ``int8k``; E4M3 values)."""
    if not fp8:
        return bhld(k_blhd), bhld(v_blhd)
    if int8k:
        kc, ks = OI.quantize_chunk_bhld(f64(k_blhd).astype(np.float32))
        kd = kc.astype(np.float64) * ks.astype(np.float64)[:, :, None, None]
    else:
        kc, ks = OF.quantize_chunk_bhld(f64(k_blhd).astype(np.float32))
        kd = OF.e4m3_decode(kc) * ks.astype(np.float64)[:, :, None, None]
    vc, vs = OF.quantize_chunk_bhld(f64(v_blhd).astype(np.float32))
    vd = OF.e4m3_decode(vc) * vs.astype(np.float64)[:, :, None, None]
    return kd, vd


def run_stream(w, ring, check_chunks, rows=None, layers=1, splits=None, device="cuda", on_check=None,
               fp8_reference="dequantised"):
    """Drive a stream through the library and the oracle.

    For each chunk: for each denoise step: for each layer: draw Q, K, V; with
    ``w.kcur_separate`` the current chunk's K/V are passed in and the KV of
    the penultimate step (the only step when there is one) is appended after
    the last step; otherwise the chunk is appended first and attention reads
    it from the ring.  At ``check_chunks`` every call is compared with the
    oracle on ``rows`` (all rows when None).  Returns the list of
    (chunk, step, layer, max|dO|, mean|dO|, max|dLSE|).
    """
    fp8 = bool(w.kv_fp8)
    i8 = bool(w.kv_int8k)
    splits = w.splits if splits is None else splits
    gen = synth.generator(w.seed)
    orings = [ListRing(w.R) for _ in range(layers)]
    orings_raw = [ListRing(w.R) for _ in range(layers)]  # un-quantised K/V (fp8 primary check)
    ws = ring.workspace(splits) if splits != 1 else None  # 0: the library's choice may split
    results = []
    if w.sink:
        sk, sv = synth.sink_kv(w, gen)
        for l in range(layers):
            ring.set_sink(l, sk.to(device), sv.to(device))
            orings[l].set_sink(*oracle_kv(sk, sv, fp8, i8))
            orings_raw[l].set_sink(bhld(sk), bhld(sv))
    rsel = slice(None) if rows is None else rows
    save_step = max(0, w.steps - 2)
    for c in range(w.chunks):
        saved = [None] * layers
        for s in range(w.steps):
            for l in range(layers):
                q, k, v = synth.chunk_qkv(w, gen)
                qd, kd, vd = q.to(device), k.to(device), v.to(device)
                if not w.kcur_separate:
                    ring.append(l, c, kd, vd)
                    orings[l].append(c, *oracle_kv(k, v, fp8, i8))
                    orings_raw[l].append(c, bhld(k), bhld(v))
                    O, LSE = ring.attention(l, c, qd, None, None, window=w.W, use_sink=w.sink,
                                            num_splits=splits, workspace=ws)
                else:
                    O, LSE = ring.attention(l, c, qd, kd, vd, window=w.W, use_sink=w.sink,
                                            num_splits=splits, workspace=ws)
                    if s == save_step:
                        saved[l] = (k, v, kd, vd)
                if c in check_chunks:
                    qq = bhld(q)[:, :, rsel]
                    kc = vc = None
                    if w.kcur_separate:
                        kc, vc = oracle_kv(k, v, False)
                    if fp8 and fp8_reference == "raw":
                        o_ref, l_ref = OA.streaming_chunk_attention(qq, orings_raw[l], c, kc, vc, w.W, w.sink,
                                                                    w.scale)
                    else:
                        o_ref, l_ref = OA.streaming_chunk_attention(qq, orings[l], c, kc, vc, w.W, w.sink,
                                                                    w.scale)
                    torch.cuda.synchronize()
                    if on_check is not None:
                        results.append((c, s, l) + on_check(O, LSE, o_ref, l_ref, rows=rows, what=f"chunk {c} step {s} layer {l}"))
        if w.kcur_separate:
            for l in range(layers):
                k, v, kd, vd = saved[l]
                ring.append(l, c, kd, vd)
                orings[l].append(c, *oracle_kv(k, v, fp8, i8))
                orings_raw[l].append(c, bhld(k), bhld(v))
    return results, orings
