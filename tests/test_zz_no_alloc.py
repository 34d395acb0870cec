"""The allocation-free chunk-attention entry point, called through the C ABI.

For callers that cannot allocate device memory (a plugin whose host
application owns all device allocations, a real-time loop that forbids
allocation after start-up), sab_chunk_attention_noalloc merges KV splits in a
library-owned device array instead of a caller workspace.  Its output must
match the regular entry point's and the oracle's on two calls in a row that
differ in queries, window and split count (the array keeps the previous
call's contents, so the second call checks that nothing stale leaks).  Collected last so that a stop at the first failure has already run
every other test; it also passes when run alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import streaming_attention_block_gb300 as sab
from oracle import attention as OA
from oracle.ring import ListRing
from streaming_attention_block_gb300 import KVRing, synth

from tests._common import bhld, compare

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _regular(lib, ring, c, q, window, splits, w, stream):
    """The regular entry point with a caller workspace (zero-filled)."""
    ws = ring.workspace(splits)
    O = torch.empty_like(q)
    L = torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda")
    st = lib.sab_chunk_attention(ring.handle, 0, c, _ptr(q), None, None, window, 1, splits, w.scale, _ptr(O),
                                 _ptr(L), _ptr(ws), ws.numel(), stream)
    assert st == 0, sab.status_string(st)
    return O, L


def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = sab.library()
    # two heads: 12 splits of 405 rows stay within the library's 8 MiB array
    w = synth.Workload("na", B=1, H=2, D=128, Lc=405, R=6, W=5, chunks=8, sink=True, kcur_separate=False, seed=71)
    gen = synth.generator(w.seed)
    ring = KVRing(1, w.B, w.H, w.D, w.Lc, w.R, has_sink=True)
    oring = ListRing(w.R)
    sk, sv = synth.sink_kv(w, gen)
    ring.set_sink(0, sk.cuda(), sv.cuda())
    oring.set_sink(bhld(sk), bhld(sv))
    qs = []
    for c in range(w.chunks):
        q, k, v = synth.chunk_qkv(w, gen)
        ring.append(0, c, k.cuda(), v.cuda())
        oring.append(c, bhld(k), bhld(v))
        qs.append(q)
    c = w.chunks - 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # Two calls in a row that differ in queries, window and split count, so
    # that partials the first call leaves in the shared array are not what
    # the second must produce: 4 splits (window 5), then 12 splits (window 4)
    # over other queries.  Each is compared with the regular entry point on
    # the same arguments and with the oracle.
    calls = [(qs[c], w.W, 4), (qs[c - 1], w.W - 1, 12)]
    for i, (q_cpu, window, splits) in enumerate(calls):
        q = q_cpu.cuda()
        O_ref, L_ref = _regular(lib, ring, c, q, window, splits, w, stream)
        O = torch.full_like(q, float("nan"))
        L = torch.full((w.B, w.H, w.Lc), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.sab_chunk_attention_noalloc(ring.handle, 0, c, _ptr(q), None, None, window, 1, splits, w.scale,
                                             _ptr(O), _ptr(L), stream)
        assert st == 0, sab.status_string(st)
        torch.cuda.synchronize()
        d = (O.float() - O_ref.float()).abs()
        assert torch.isfinite(O.float()).all(), f"call {i}: non-finite output"
        assert d.max().item() <= 1e-2 and d.mean().item() <= 1e-3, f"call {i}: max {d.max().item():.3e}"
        assert (L - L_ref).abs().max().item() <= 1e-3, f"call {i}"
        o_or, l_or = OA.streaming_chunk_attention(bhld(q_cpu), oring, c, None, None, window, True, w.scale)
        compare(O, L, o_or, l_or, what=f"no-alloc call {i} vs oracle")
    # a request larger than the library's scratch is refused before any launch
    big = synth.Workload("nb", B=2, H=24, D=128, Lc=1536, R=2, W=1, seed=72)
    rbig = KVRing(1, big.B, big.H, big.D, big.Lc, big.R)
    qb, kb, vb = (x.cuda() for x in synth.chunk_qkv(big, synth.generator(big.seed)))
    Ob = torch.empty_like(qb)
    st = lib.sab_chunk_attention_noalloc(rbig.handle, 0, 0, _ptr(qb), _ptr(kb), _ptr(vb), 1, 0, 8, big.scale,
                                         _ptr(Ob), None, stream)
    assert st == 4  # SAB_ERR_WORKSPACE
    assert lib.sab_get_last_device_error(stream) == 0
