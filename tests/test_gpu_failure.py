"""Failure detection without a GPU fault: a device pipeline wait that nothing
completes gives up after its limit, the host reads SAB_ERR_TIMEOUT, the record
clears, and the context keeps working (a streaming call afterwards still
matches the oracle).  Nothing here faults, traps or hangs a GPU."""

import time

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle.ring import ListRing
from streaming_attention_block_gb300 import KVRing, synth
import streaming_attention_block_gb300 as sab

from tests._common import bhld, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


def test_bounded_wait_gives_up_and_context_survives():
    assert sab.get_last_device_error() == 0
    t0 = time.perf_counter()
    sab.selftest_bounded_wait(50_000_000)  # 50 ms
    status = sab.get_last_device_error()
    elapsed = time.perf_counter() - t0
    assert status == 6, sab.status_string(status)  # SAB_ERR_TIMEOUT
    assert elapsed >= 0.045  # the wait really waited for its limit
    assert sab.get_last_device_error() == 0  # the record was cleared

    # the context is still usable: one streaming call against the oracle
    w = synth.Workload("f", B=1, H=2, D=128, Lc=256, R=2, W=2, seed=81)
    ring = KVRing(1, w.B, w.H, w.D, w.Lc, w.R)
    oring = ListRing(w.R)
    gen = synth.generator(w.seed)
    for c in range(3):
        q, k, v = synth.chunk_qkv(w, gen)
        O, L = ring.attention(0, c, q.cuda(), k.cuda(), v.cuda(), window=w.W, num_splits=1)
        o_ref, l_ref = OA.streaming_chunk_attention(bhld(q), oring, c, bhld(k), bhld(v), w.W, False, w.scale)
        torch.cuda.synchronize()
        compare(O, L, o_ref, l_ref, what=f"after timeout, chunk {c}")
        ring.append(0, c, k.cuda(), v.cuda())
        oring.append(c, bhld(k), bhld(v))
    assert sab.get_last_device_error() == 0


def test_selftest_rejects_limits_outside_range():
    with pytest.raises(sab.SabError):
        sab.selftest_bounded_wait(10)
    with pytest.raises(sab.SabError):
        sab.selftest_bounded_wait(5_000_000_000)


def test_split_abort_leaves_workspace_usable():
    """A split call whose merge sees one aborted split (the self-test hook:
    that split reports itself exactly as a split whose wait gave up) skips
    the merge, reports SAB_ERR_TIMEOUT and leaves every arrival counter of
    the caller's workspace at zero; the next split call on the same
    workspace, without re-zeroing it, matches the oracle."""
    w = synth.Workload("fa", B=1, H=3, D=128, Lc=300, R=3, W=2, chunks=4, sink=True, kcur_separate=False, seed=82)
    ring = KVRing(1, w.B, w.H, w.D, w.Lc, w.R, has_sink=True)
    oring = ListRing(w.R)
    gen = synth.generator(w.seed)
    sk, sv = synth.sink_kv(w, gen)
    ring.set_sink(0, sk.cuda(), sv.cuda())
    oring.set_sink(bhld(sk), bhld(sv))
    splits = 12  # merged through the workspace, the last arriver by atomic ticket; some splits empty
    ws = ring.workspace(splits)
    n_counters = w.B * w.H * 3  # one per (b, h) and 128-row query tile: 300 rows = 3 tiles
    for c in range(w.chunks):
        q, k, v = synth.chunk_qkv(w, gen)
        ring.append(0, c, k.cuda(), v.cuda())
        oring.append(c, bhld(k), bhld(v))
        O = torch.empty((w.B, w.Lc, w.H, w.D), dtype=torch.bfloat16, device="cuda")
        L = torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda")
        if c % 2 == 0:
            sab.selftest_split_abort(ring.handle, 0, c, q.cuda(), None, None, w.W, True, splits, w.scale, O, L, ws,
                                     abort_split=c % splits)
            assert sab.get_last_device_error() == 6  # SAB_ERR_TIMEOUT
            assert sab.get_last_device_error() == 0
            assert int(ws[:4 * n_counters].view(torch.int32).abs().sum().item()) == 0, "counters left non-zero"
        sab.chunk_attention(ring.handle, 0, c, q.cuda(), None, None, w.W, True, splits, w.scale, O, L, ws)
        o_ref, l_ref = OA.streaming_chunk_attention(bhld(q), oring, c, None, None, w.W, True, w.scale)
        torch.cuda.synchronize()
        compare(O, L, o_ref, l_ref, what=f"split call after an aborted one, chunk {c}")
        assert sab.get_last_device_error() == 0
    with pytest.raises(sab.SabError):  # the hook needs a split call (>= 2 splits)
        sab.selftest_split_abort(ring.handle, 0, w.chunks - 1, q.cuda(), None, None, w.W, True, 1, w.scale, O, L, ws,
                                 abort_split=0)
