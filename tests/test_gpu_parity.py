"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Element-by-element on small workloads that span several tiles and a ragged
tail; on sampled outputs at the full workload sizes, in the launch
configuration the bench times.  Ring contents after append are compared bit
for bit with the slots the list ring implies.
"""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import ring as OR
from oracle.ring import expected_physical_slots
from streaming_attention_block_gb300 import KVRing, SabError, synth
import streaming_attention_block_gb300 as sab

from tests._common import bhld, compare, f32, f64, run_stream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()
    torch.cuda.init()


def _ring(w, layers=1):
    return KVRing(layers, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink,
                  kv_dtype=sab.KV_FP8_E4M3 if w.kv_fp8 else sab.KV_BF16)


def _check_device_error():
    assert sab.get_last_device_error() == 0


# --------------------------------------------------------------- ring / append

@pytest.mark.parametrize("B,H,D,Lc,R,sink", [(1, 2, 64, 32, 2, False), (2, 3, 128, 200, 3, True),
                                             (1, 4, 128, 405, 5, True)])
def test_append_bf16_bit_exact(B, H, D, Lc, R, sink):
    w = synth.Workload("t", B=B, H=H, D=D, Lc=Lc, R=R, W=1, chunks=3 * R + 1, sink=sink, seed=7)
    ring = _ring(w)
    gen = synth.generator(7)
    from oracle.ring import ListRing
    lr = ListRing(R)
    rows0 = int(sink) * Lc
    if sink:
        sk, sv = synth.sink_kv(w, gen)
        ring.set_sink(0, sk.cuda(), sv.cuda())
    zeros = np.zeros((R, B, H, Lc, D), dtype=np.int16)
    for c in range(w.chunks):
        _, k, v = synth.chunk_qkv(w, gen)
        ring.append(0, c, k.cuda(), v.cuda())
        lr.append(c, k.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy(),
                  v.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy())
        if c == 1:  # an in-place rewrite of the newest chunk
            _, k2, v2 = synth.chunk_qkv(w, gen)
            ring.append(0, c, k2.cuda(), v2.cuda())
            lr.append(c, k2.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy(),
                      v2.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy())
        torch.cuda.synchronize()
        K, V, _, _ = ring.layer_views(0)
        Kb = K.view(torch.int16).cpu().numpy()
        Vb = V.view(torch.int16).cpu().numpy()
        for which, got in ((0, Kb), (1, Vb)):
            exp = expected_physical_slots(lr, zeros, which)
            for r in range(R):
                seg = got[:, :, rows0 + r * Lc: rows0 + (r + 1) * Lc]
                assert np.array_equal(seg, exp[r]), f"chunk {c} slot {r} tensor {which}"
        if sink:
            assert np.array_equal(Kb[:, :, :Lc], sk.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy())
            assert np.array_equal(Vb[:, :, :Lc], sv.permute(0, 2, 1, 3).contiguous().view(torch.int16).numpy())
        held = lr.held_chunks()
        for x in held:
            assert ring.slot_of(0, x) == x % R
        with pytest.raises(SabError):
            ring.slot_of(0, c + 1)
        if held[0] > 0:
            with pytest.raises(SabError):
                ring.slot_of(0, held[0] - 1)


def test_append_order_and_state():
    w = synth.Workload("t", B=1, H=2, D=64, Lc=32, R=2, seed=3)
    ring = _ring(w, layers=2)
    _, k, v = synth.chunk_qkv(w, synth.generator(3))
    k, v = k.cuda(), v.cuda()
    ring.append(0, 5, k, v)  # a stream may start at any chunk
    with pytest.raises(SabError) as e:
        ring.append(0, 7, k, v)
    assert e.value.status == 3
    with pytest.raises(SabError):
        ring.append(0, 4, k, v)
    ring.append(0, 6, k, v)
    ring.append(0, 7, k, v)
    # the held chunks map to slot chunk mod R; older, newer or never-appended
    # chunks are OUT_OF_RANGE (the oracle's ring model: slot_of)
    assert ring.slot_of(0, 7) == OR.slot_of(7, w.R) and ring.slot_of(0, 6) == OR.slot_of(6, w.R)
    for layer, chunk in ((0, 5), (0, 8), (1, 0)):
        with pytest.raises(SabError) as e:
            ring.slot_of(layer, chunk)
        assert e.value.status == 3
    n, h, s = sab.kv_ring_get_state(ring.handle, 2)
    assert n == [7, -1] and h == [2, 0] and s == [0, 0]
    sab.kv_ring_set_state(ring.handle, [3, 0], [2, 1], [0, 0])
    assert sab.kv_ring_get_state(ring.handle, 2) == ([3, 0], [2, 1], [0, 0])
    with pytest.raises(SabError):
        sab.kv_ring_set_state(ring.handle, [3, 0], [3, 1], [0, 0])  # held > R
    with pytest.raises(SabError):
        ring.set_sink(0, k, v)  # no sink slot
    torch.cuda.synchronize()


# ------------------------------------------------------------ attention: small

SMALL = [
    # name, workload overrides, splits
    ("tiny", synth.workload("tiny"), 1),
    ("tiny_split3", synth.workload("tiny"), 3),
    ("ragged_sink_kcur", synth.Workload("rk", B=2, H=3, D=128, Lc=200, R=3, W=2, chunks=7, sink=True, seed=11), 1),
    ("ragged_sink_kcur_split3", synth.Workload("rk", B=2, H=3, D=128, Lc=200, R=3, W=2, chunks=7, sink=True,
                                               seed=12), 3),
    ("ring_current_in_ring", synth.Workload("rr", B=1, H=2, D=128, Lc=300, R=4, W=3, chunks=10, sink=True,
                                            kcur_separate=False, seed=13), 4),
    ("d64_window1", synth.Workload("d64", B=1, H=3, D=64, Lc=160, R=2, W=1, chunks=5, seed=14), 1),
    ("window0_R1", synth.Workload("w0", B=1, H=2, D=128, Lc=130, R=1, W=0, chunks=3, seed=15), 2),
    # the sink and the current chunk only (window 0), current chunk passed in / appended first
    ("sink_window0_kcur", synth.Workload("sw0", B=2, H=2, D=64, Lc=96, R=1, W=0, chunks=4, sink=True, seed=17), 1),
    ("sink_window0_in_ring", synth.Workload("sw1", B=1, H=3, D=128, Lc=200, R=1, W=0, chunks=4, sink=True,
                                            kcur_separate=False, seed=18), 3),
    ("many_empty_splits", synth.Workload("es", B=1, H=2, D=128, Lc=96, R=2, W=2, chunks=4, seed=16), 9),
]


@pytest.mark.parametrize("name,w,splits", SMALL, ids=[s[0] for s in SMALL])
def test_streaming_small_elementwise(name, w, splits):
    ring = _ring(w)
    res, _ = run_stream(w, ring, check_chunks=set(range(w.chunks)), splits=splits, on_check=compare)
    assert len(res) == w.chunks * w.steps
    _check_device_error()


@pytest.mark.parametrize("Lc,W,L_chunks,H,D,splits", [(200, 2, 5, 2, 128, 1), (256, 2, 6, 2, 128, 2),
                                                      (128, 1, 7, 3, 64, 1), (96, 3, 5, 1, 128, 3),
                                                      (160, 0, 4, 2, 128, 1),   # chunk-local only
                                                      (64, 8, 5, 2, 64, 2)])   # window past the start: causal
def test_block_causal_small_elementwise(Lc, W, L_chunks, H, D, splits):
    w = synth.Workload("bc", B=2, H=H, D=D, Lc=Lc, W=W, seq_chunks=L_chunks, seed=21)
    q, k, v = synth.full_sequence_qkv(w, synth.generator(21))
    L = L_chunks * Lc
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    O = torch.empty_like(qd)
    LSE = torch.empty((2, H, L), dtype=torch.float32, device="cuda")
    n = sab.block_causal_attention_workspace(2, L, H, D, splits)
    ws = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda") if n else None
    sab.block_causal_attention(qd, kd, vd, Lc, W, splits, D ** -0.5, O, LSE, ws)
    torch.cuda.synchronize()
    o_ref, l_ref = OA.block_causal_attention(f64(q), f64(k), f64(v), Lc, W, D ** -0.5)
    compare(O, LSE, o_ref, l_ref, what=f"block-causal Lc={Lc}")
    _check_device_error()


def test_splits_equal_unsplit():
    """Split-KV + in-kernel LSE merge equals the unsplit kernel (any size)."""
    w = synth.Workload("sp", B=1, H=4, D=128, Lc=405, R=6, W=5, chunks=8, sink=True, kcur_separate=False, seed=31)
    gen = synth.generator(31)
    ring = _ring(w)
    sk, sv = synth.sink_kv(w, gen)
    ring.set_sink(0, sk.cuda(), sv.cuda())
    for c in range(w.chunks):
        q, k, v = (x.cuda() for x in synth.chunk_qkv(w, gen))
        ring.append(0, c, k, v)
    O1, L1 = ring.attention(0, w.chunks - 1, q, window=w.W, use_sink=True, num_splits=1)
    for s in (2, 5, 8, 40):
        Os, Ls = ring.attention(0, w.chunks - 1, q, window=w.W, use_sink=True, num_splits=s)
        torch.cuda.synchronize()
        assert (Os.float() - O1.float()).abs().max().item() <= 8e-3
        assert (Ls - L1).abs().max().item() <= 1e-4
    _check_device_error()


def test_api_errors_launch_nothing():
    w = synth.Workload("e", B=1, H=2, D=128, Lc=64, R=2, W=2, seed=41)
    ring = _ring(w)
    q, k, v = (x.cuda() for x in synth.chunk_qkv(w, synth.generator(41)))
    O = torch.full_like(q, 7.0)
    # chunk 1 needs chunk 0, never appended
    with pytest.raises(SabError) as e:
        ring.attention(0, 1, q, k, v, window=2, O=O)
    assert e.value.status == 3
    # no K_cur and the chunk is not in the ring
    with pytest.raises(SabError):
        ring.attention(0, 0, q, window=2, O=O)
    # sink requested on a ring without a sink
    with pytest.raises(SabError):
        ring.attention(0, 0, q, k, v, window=2, use_sink=True, O=O)
    # split without workspace
    with pytest.raises(SabError) as e:
        sab.chunk_attention(ring.handle, 0, 0, q, k, v, 2, False, 4, 0.1, O, None, None)
    assert e.value.status == 4
    # misaligned pointer
    with pytest.raises(SabError):
        sab.chunk_attention(ring.handle, 0, 0, q.data_ptr() + 2, k, v, 2, False, 1, 0.1, O, None, None)
    # window eviction: ring of 2 holds chunks 1, 2; window 3 at chunk 3 needs chunk 0
    for c in range(3):
        ring.append(0, c, k, v)
    with pytest.raises(SabError):
        ring.attention(0, 3, q, k, v, window=3, O=O)
    torch.cuda.synchronize()
    assert torch.all(O.float() == 7.0)  # nothing was written
    ring.attention(0, 3, q, k, v, window=2, O=O)
    torch.cuda.synchronize()
    assert not torch.all(O.float() == 7.0)
    _check_device_error()


# ------------------------------------------------------- attention: full sizes

def test_wan13b_stream_sampled_rows():
    """Wan-1.3B shape (H12 D128 Lc1536, ring 2, window 2, 4 steps) on layer 0:
    every call of chunks 0-3 and 19 compared on a sample of query rows."""
    w = synth.workload("wan13b", layers=1)
    ring = _ring(w)
    rows = np.concatenate([np.arange(0, 1536, 7), [1535]])
    res, _ = run_stream(w, ring, check_chunks={0, 1, 2, 3, 19}, rows=rows, on_check=compare)
    assert len(res) == 5 * 4
    _check_device_error()


def test_long_sink_stream_sampled_rows():
    """Sink + 20-slot ring, 405 tokens per chunk, 60 chunks (3 wraps), 8 KV
    splits merged in-kernel; checked around every wrap boundary."""
    w = synth.workload("long_sink")
    ring = _ring(w)
    rows = np.concatenate([np.arange(0, 405, 5), [383, 384, 404]])
    res, _ = run_stream(w, ring, check_chunks={0, 1, 18, 19, 20, 21, 39, 40, 59}, rows=rows, on_check=compare)
    assert len(res) == 9
    _check_device_error()


def test_long_sink_stream_auto_sampled_rows():
    """The same stream through the library's own launch choice
    (num_splits = 0, the configuration the benchmark times), checked at the
    chunks on both sides of every wrap."""
    w = synth.workload("long_sink")
    ring = _ring(w)
    rows = np.concatenate([np.arange(0, 405, 5), [383, 384, 404]])
    res, _ = run_stream(w, ring, check_chunks={0, 1, 18, 19, 20, 21, 39, 40, 59}, rows=rows, splits=0, on_check=compare)
    assert len(res) == 9
    _check_device_error()


def test_block_causal_full_size_rows():
    """B2 x 30720 tokens, H12, D128, window 2, every head: in batch 0 four
    rows of every one of the 240 query tiles (its first and last row and two
    drawn at random); in batch 1, 512 random rows of every chunk."""
    w = synth.workload("block_causal")
    q, k, v = synth.full_sequence_qkv(w, synth.generator(w.seed))
    L = w.seq_chunks * w.Lc
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    O = torch.empty_like(qd)
    LSE = torch.empty((w.B, w.H, L), dtype=torch.float32, device="cuda")
    sab.block_causal_attention(qd, kd, vd, w.Lc, w.W, 0, w.scale, O, LSE, None)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    tiles = L // 128
    rows0 = np.unique(np.concatenate([np.arange(tiles) * 128, np.arange(tiles) * 128 + 127,
                                      np.arange(tiles) * 128 + rng.integers(1, 127, tiles),
                                      np.arange(tiles) * 128 + rng.integers(1, 127, tiles)]))
    assert len(np.unique(rows0 // 128)) == tiles
    rows1 = np.unique(np.concatenate([c * w.Lc + rng.choice(w.Lc, 512, replace=False) for c in range(w.seq_chunks)]))
    qf, kf, vf = f32(q), f32(k), f32(v)
    for b, rows in ((0, rows0), (1, rows1)):
        o_ref, l_ref = OA.block_causal_attention(qf, kf, vf, w.Lc, w.W, w.scale, rows=rows, batches=[b])
        compare(O[b:b + 1], LSE[b:b + 1], o_ref, l_ref, rows=rows, what=f"block-causal full, batch {b}")
    _check_device_error()
