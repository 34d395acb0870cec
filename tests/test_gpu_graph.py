"""GPU checks of the graph-capturable streaming calls (chunk index read from
device memory): they plan the same key sets on the device as the host calls
do on the host -- outputs bit-identical to sab_chunk_attention on the same
inputs, unsplit and split, BF16 and FP8 rings -- and one chunk step captured
in a CUDA graph replays correctly for every later chunk: bit-identical to the
host-indexed calls, and within the parity tolerances of the CPU oracle on
every replay across several ring wraps (current chunk passed in, or written
into its slot first behind a sink; BF16 and E4M3 rings)."""

import pytest
import torch

from oracle import attention as OA
from oracle.ring import ListRing
from streaming_attention_block_gb300 import KVRing, synth
import streaming_attention_block_gb300 as sab

from tests._common import FP8_LSE, FP8_MAX, bhld, compare, oracle_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


def _kv_dtype(w):
    return (sab.KV_INT8K_FP8V if w.kv_int8k else sab.KV_FP8_E4M3) if w.kv_fp8 else sab.KV_BF16


def _rings(w, layers):
    mk = lambda: KVRing(layers, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=_kv_dtype(w))
    return mk(), mk()


def _drive(w, layers, splits, step_fn):
    """Run w.chunks chunks; step_fn(c, s, l, q, k, v, save) does both paths."""
    gen = synth.generator(w.seed)
    for c in range(w.chunks):
        for s in range(w.steps):
            for l in range(layers):
                q, k, v = (x.cuda() for x in synth.chunk_qkv(w, gen))
                step_fn(c, s, l, q, k, v)


CASES = [
    ("bf16_kcur_unsplit", synth.Workload("g", B=1, H=2, D=128, Lc=256, R=2, W=2, chunks=6, steps=2, seed=71), 1),
    ("bf16_kcur_split2", synth.Workload("g", B=1, H=3, D=128, Lc=384, R=3, W=3, chunks=7, steps=2, seed=72), 2),
    ("bf16_sink_inring", synth.Workload("g", B=2, H=2, D=64, Lc=200, R=4, W=3, chunks=9, sink=True,
                                        kcur_separate=False, seed=73), 1),
    ("fp8_sink_inring_split3", synth.Workload("g", B=1, H=2, D=128, Lc=160, R=4, W=3, chunks=9, sink=True,
                                              kcur_separate=False, kv_fp8=True, outliers=True, seed=74), 3),
]


@pytest.mark.parametrize("name,w,splits", CASES, ids=[c[0] for c in CASES])
def test_dev_calls_match_host_calls(name, w, splits):
    layers = 2
    rh, rd = _rings(w, layers)
    d_chunk = torch.zeros(1, dtype=torch.int64, device="cuda")
    wsh, wsd = rh.workspace(splits) if splits > 1 else None, rd.workspace(splits) if splits > 1 else None
    if w.sink:
        sk, sv = (x.cuda() for x in synth.sink_kv(w, synth.generator(w.seed + 1)))
        for l in range(layers):
            rh.set_sink(l, sk, sv)
            rd.set_sink(l, sk, sv)
    save = max(0, w.steps - 2)
    saved = {}
    shape = (w.B, w.Lc, w.H, w.D)

    def step(c, s, l, q, k, v):
        if not w.kcur_separate:
            rh.append(l, c, k, v)
            sab.kv_ring_append_dev(rd.handle, l, d_chunk, k, v)
        kc, vc = (k, v) if w.kcur_separate else (None, None)
        Oh, Lh = rh.attention(l, c, q, kc, vc, window=w.W, use_sink=w.sink, num_splits=splits, workspace=wsh)
        Od = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        Ld = torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda")
        sab.chunk_attention_dev(rd.handle, l, d_chunk, q, kc, vc, w.W, w.sink, splits, w.scale, Od, Ld, wsd)
        assert torch.equal(Oh, Od), f"{name}: chunk {c} step {s} layer {l}: O differs"
        assert torch.equal(Lh, Ld), f"{name}: chunk {c} step {s} layer {l}: LSE differs"
        if w.kcur_separate and s == save:
            saved[l] = (k, v)
        if l == layers - 1 and s == w.steps - 1:
            if w.kcur_separate:
                for ll in range(layers):
                    rh.append(ll, c, *saved[ll])
                    sab.kv_ring_append_dev(rd.handle, ll, d_chunk, *saved[ll])
            sab.chunk_counter_add(d_chunk, 1)

    _drive(w, layers, splits, step)
    torch.cuda.synchronize()
    assert int(d_chunk.item()) == w.chunks
    assert sab.get_last_device_error() == 0


def test_graph_replay_matches_host_calls():
    """Capture one chunk step (2 denoise steps x 2 layers of attention, the
    appends and the counter advance) once; replay it for chunks 0..7 with
    fresh inputs copied into the captured buffers; compare every output with
    the host-indexed calls on a second ring."""
    w = synth.Workload("g", B=1, H=4, D=128, Lc=512, R=2, W=2, chunks=8, steps=2, seed=75)
    layers, S = 2, w.steps
    rh, rd = _rings(w, layers)
    shape = (w.B, w.Lc, w.H, w.D)
    bufs = {(s, l): [torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
            for s in range(S) for l in range(layers)}
    outs = {(s, l): (torch.empty(shape, dtype=torch.bfloat16, device="cuda"),
                     torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda"))
            for s in range(S) for l in range(layers)}
    d_chunk = torch.zeros(1, dtype=torch.int64, device="cuda")
    save = max(0, S - 2)
    # warm up the kernels' one-time attribute setup outside the capture
    q0, k0, v0 = bufs[(0, 0)]
    for t in (q0, k0, v0):
        t.normal_()
    rh.attention(0, 0, q0, k0, v0, window=w.W, num_splits=1)
    torch.cuda.synchronize()
    rh, _ = _rings(w, layers)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        for s in range(S):
            for l in range(layers):
                q, k, v = bufs[(s, l)]
                O, L = outs[(s, l)]
                sab.chunk_attention_dev(rd.handle, l, d_chunk, q, k, v, w.W, False, 1, w.scale, O, L, None, st)
        for l in range(layers):
            _, k, v = bufs[(save, l)]
            sab.kv_ring_append_dev(rd.handle, l, d_chunk, k, v, st)
        sab.chunk_counter_add(d_chunk, 1, st)
    torch.cuda.synchronize()
    d_chunk.zero_()  # capture does not run the work

    gen = synth.generator(w.seed)
    for c in range(w.chunks):
        fresh = {}
        for s in range(S):
            for l in range(layers):
                fresh[(s, l)] = [x.cuda() for x in synth.chunk_qkv(w, gen)]
                for dst, src in zip(bufs[(s, l)], fresh[(s, l)]):
                    dst.copy_(src)
        g.replay()
        for s in range(S):
            for l in range(layers):
                q, k, v = fresh[(s, l)]
                Oh, Lh = rh.attention(l, c, q, k, v, window=w.W, num_splits=1)
                O, L = outs[(s, l)]
                assert torch.equal(Oh, O), f"chunk {c} step {s} layer {l}: O differs after replay"
                assert torch.equal(Lh, L), f"chunk {c} step {s} layer {l}: LSE differs after replay"
        for l in range(layers):
            _, k, v = fresh[(save, l)]
            rh.append(l, c, k, v)
    torch.cuda.synchronize()
    assert int(d_chunk.item()) == w.chunks
    assert sab.get_last_device_error() == 0


# Graph replay against the CPU oracle ("Matrix-Game 4.0", section
# 前置知识 / FP8 量化与 CUDA Graph: one recorded chunk step replayed per chunk).
# Each case streams past several ring wraps; every replay's outputs (every
# denoise step and layer, all rows) are compared with the oracle's list ring.
ORACLE_CASES = [
    # current chunk passed in, KV of the penultimate step appended after the steps
    ("kcur_3wraps", synth.Workload("go", B=1, H=2, D=128, Lc=256, R=2, W=2, chunks=7, steps=2, seed=91)),
    # sink + current chunk written into its slot first (ragged 200-token chunks)
    ("sink_inring_ragged", synth.Workload("go", B=1, H=2, D=128, Lc=200, R=4, W=3, chunks=10, steps=2, sink=True,
                                          kcur_separate=False, seed=92)),
    # E4M3 ring, sink, current chunk in the ring, outliers
    ("fp8_sink_inring", synth.Workload("go", B=1, H=2, D=128, Lc=160, R=3, W=2, chunks=8, steps=1, sink=True,
                                       kcur_separate=False, kv_fp8=True, outliers=True, seed=93)),
    # INT8 keys / E4M3 values, sink, current chunk in the ring
    ("int8k_sink_inring", synth.Workload("go", B=1, H=2, D=128, Lc=160, R=3, W=2, chunks=8, steps=1, sink=True,
                                         kcur_separate=False, kv_fp8=True, kv_int8k=True, outliers=True, seed=94)),
    # a window shorter than the ring: the device planner takes the newest chunks only
    ("kcur_window1_R4", synth.Workload("go", B=1, H=2, D=128, Lc=192, R=4, W=1, chunks=9, steps=1, seed=95)),
]


@pytest.mark.parametrize("name,w", ORACLE_CASES, ids=[c[0] for c in ORACLE_CASES])
def test_graph_replay_matches_oracle(name, w):
    layers, S = 2, w.steps
    fp8 = bool(w.kv_fp8)
    int8k = bool(w.kv_int8k)
    shape = (w.B, w.Lc, w.H, w.D)
    mk = lambda: KVRing(layers, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=_kv_dtype(w))
    # one-time kernel attribute set-up happens outside the capture
    scratch = mk()
    if w.sink:
        zs = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        scratch.set_sink(0, zs, zs)
    z = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    scratch.append(0, 0, z, z)
    scratch.attention(0, 0, z, None if not w.kcur_separate else z, None if not w.kcur_separate else z,
                      window=w.W, use_sink=w.sink, num_splits=1)
    torch.cuda.synchronize()
    del scratch

    ring = mk()
    orings = [ListRing(w.R) for _ in range(layers)]
    gen = synth.generator(w.seed)
    if w.sink:
        sk, sv = synth.sink_kv(w, gen)
        for l in range(layers):
            ring.set_sink(l, sk.cuda(), sv.cuda())
            orings[l].set_sink(*oracle_kv(sk, sv, fp8, int8k))
    bufs = {(s, l): [torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
            for s in range(S) for l in range(layers)}
    outs = {(s, l): (torch.empty(shape, dtype=torch.bfloat16, device="cuda"),
                     torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda"))
            for s in range(S) for l in range(layers)}
    d_chunk = torch.zeros(1, dtype=torch.int64, device="cuda")
    save = max(0, S - 2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        for s in range(S):
            for l in range(layers):
                q, k, v = bufs[(s, l)]
                O, L = outs[(s, l)]
                if not w.kcur_separate:
                    sab.kv_ring_append_dev(ring.handle, l, d_chunk, k, v, st)
                    sab.chunk_attention_dev(ring.handle, l, d_chunk, q, None, None, w.W, w.sink, 1, w.scale, O, L,
                                            None, st)
                else:
                    sab.chunk_attention_dev(ring.handle, l, d_chunk, q, k, v, w.W, w.sink, 1, w.scale, O, L, None, st)
        if w.kcur_separate:
            for l in range(layers):
                _, k, v = bufs[(save, l)]
                sab.kv_ring_append_dev(ring.handle, l, d_chunk, k, v, st)
        sab.chunk_counter_add(d_chunk, 1, st)
    torch.cuda.synchronize()
    d_chunk.zero_()  # capture does not run the work

    def check(O, L, o_ref, l_ref, what):
        if fp8:
            return compare(O, L, o_ref, l_ref, max_tol=FP8_MAX, mean_tol=2e-3, lse_tol=FP8_LSE, what=what,
                           rel_ulp=2.0 ** -8)
        return compare(O, L, o_ref, l_ref, what=what)

    for c in range(w.chunks):
        host = {}
        for s in range(S):
            for l in range(layers):
                host[(s, l)] = synth.chunk_qkv(w, gen)
                for dst, src in zip(bufs[(s, l)], host[(s, l)]):
                    dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        for s in range(S):
            for l in range(layers):
                q, k, v = host[(s, l)]
                if not w.kcur_separate:
                    orings[l].append(c, *oracle_kv(k, v, fp8, int8k))
                    o_ref, l_ref = OA.streaming_chunk_attention(bhld(q), orings[l], c, None, None, w.W, w.sink,
                                                                w.scale)
                else:
                    kc, vc = oracle_kv(k, v, False)
                    o_ref, l_ref = OA.streaming_chunk_attention(bhld(q), orings[l], c, kc, vc, w.W, w.sink, w.scale)
                O, L = outs[(s, l)]
                check(O, L, o_ref, l_ref, f"{name}: replay of chunk {c}, step {s}, layer {l}")
        if w.kcur_separate:
            for l in range(layers):
                _, k, v = host[(save, l)]
                orings[l].append(c, *oracle_kv(k, v, fp8, int8k))
    assert int(d_chunk.item()) == w.chunks
    assert sab.get_last_device_error() == 0

