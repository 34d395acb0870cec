"""Debug build (libsab_debug.so, compiled with -DSAB_DEBUG_BOUNDS): device-side
index checks that record SAB_ERR_BOUNDS and leave the kernel before any copy or
store, never trapping.

``test_small_cases_under_debug_build`` re-runs the small GPU cases in a child
process with the debug library loaded (``SAB_LIBRARY``): every index check
passes on valid calls, the results still match the oracle, and the canary
bands around rings and workspaces stay intact (the conftest fixture checks
them after every GPU test).  The injection tests run only in that child: each
forges one index past its buffer from the host and checks that the device
check catches it -- the error word reads SAB_ERR_BOUNDS, no byte of the ring,
the output or the canaries changed, and the next call on the same ring and
workspace is correct again.  The forged indices point inside memory the test
owns (one slot past the ring rows lands in the canary band after the ring; a
key run past the ring is read by tensor copies that fill zeros out of range;
the workspace bound is lowered, not overrun), so nothing can fault even if a
check were missing.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle.ring import ListRing
from streaming_attention_block_gb300 import KVRing, synth
import streaming_attention_block_gb300 as sab

from tests._common import bhld, compare

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHILD = os.environ.get("SAB_DEBUG_BOUNDS_CHILD") == "1"
# small cases of every kernel: BF16 / 8-bit appends, streaming (split and
# unsplit, sink, current chunk passed in), block-causal, memory prefix,
# backward, graph-mode device plans, fused rope + append, failure paths
SMALL_CASES = ("bit_exact or append_order or streaming_small or block_causal_small or splits_equal_unsplit "
               "or fp8_attention_small or int8k_attention_small or fp8mma_small or dev_calls "
               "or graph_replay_matches_oracle or memory_prefix_elementwise or backward_matches_oracle "
               "or qk_norm_rope or fused_append or split_abort or bounded_wait or injected")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


@pytest.mark.skipif(CHILD, reason="runs in the parent process only")
def test_small_cases_under_debug_build():
    from streaming_attention_block_gb300.build import DEBUG_LIB, build
    build(debug_bounds=True)
    env = dict(os.environ, SAB_LIBRARY=DEBUG_LIB, SAB_DEBUG_BOUNDS_CHILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-rs", "-m", "gpu", "-k", SMALL_CASES, "-p",
                        "no:cacheprovider", os.path.join(ROOT, "tests")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    out = r.stdout + r.stderr
    tail = "\n".join(out.splitlines()[-25:])
    assert r.returncode == 0, tail
    assert " passed" in tail, tail
    assert "debug-build child" not in out, tail  # the injection tests ran there


needs_debug = pytest.mark.skipif(not CHILD, reason="runs in the debug-build child process")


def _stream_ring(w, chunks, kv_dtype=sab.KV_BF16):
    """A ring holding chunks 0 .. chunks - 1, and the oracle's copy."""
    ring = KVRing(1, w.B, w.H, w.D, w.Lc, w.R, kv_dtype=kv_dtype)
    oring = ListRing(w.R)
    gen = synth.generator(w.seed)
    for c in range(chunks):
        q, k, v = synth.chunk_qkv(w, gen)
        ring.append(0, c, k.cuda(), v.cuda())
        oring.append(c, bhld(k), bhld(v))
    return ring, oring, gen


@needs_debug
@pytest.mark.parametrize("kv_dtype", [sab.KV_BF16, sab.KV_FP8_E4M3, sab.KV_INT8K_FP8V], ids=["bf16", "fp8", "int8k"])
def test_injected_append_slot_is_caught(kv_dtype):
    assert sab.debug_bounds_enabled()
    w = synth.Workload("dbg_append", B=1, H=2, D=128, Lc=128, R=2, W=1, seed=91)
    ring, _, gen = _stream_ring(w, 2, kv_dtype)
    torch.cuda.synchronize()
    before = ring.mem.clone()
    sab.debug_inject_bounds_error(sab.DEBUG_INJECT_APPEND_SLOT)
    q, k, v = synth.chunk_qkv(w, gen)
    ring.append(0, 2, k.cuda(), v.cuda())  # the host accepts it; the device check refuses the slot
    assert sab.get_last_device_error() == sab.ERR_BOUNDS
    assert torch.equal(ring.mem, before), "an append that failed its index check wrote memory"
    # the next append is a normal one and writes its slot
    ring.append(0, 3, k.cuda(), v.cuda())
    assert sab.get_last_device_error() == 0
    assert not torch.equal(ring.mem, before)


@needs_debug
@pytest.mark.parametrize("splits", [1, 3])
def test_injected_key_row_is_caught(splits):
    """Every CTA whose key tiles include the forged run leaves before any copy;
    with one split that is every CTA (O and LSE untouched), with three the
    merge of every query tile sees an aborted split and stores nothing."""
    w = synth.Workload("dbg_key", B=1, H=2, D=128, Lc=256, R=2, W=2, seed=92)
    ring, oring, gen = _stream_ring(w, 2)
    q, k, v = synth.chunk_qkv(w, gen)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = ring.workspace(splits) if splits > 1 else None
    O = torch.full_like(qd, 7.0)
    LSE = torch.full((w.B, w.H, w.Lc), 7.0, dtype=torch.float32, device="cuda")
    sab.debug_inject_bounds_error(sab.DEBUG_INJECT_KEY_ROW)
    ring.attention(0, 2, qd, kd, vd, window=w.W, num_splits=splits, O=O, LSE=LSE, workspace=ws)
    assert sab.get_last_device_error() == sab.ERR_BOUNDS
    assert bool((O == 7.0).all()) and bool((LSE == 7.0).all())
    # the same ring and workspace (counters back at zero) give the right answer next
    O, LSE = ring.attention(0, 2, qd, kd, vd, window=w.W, num_splits=splits, workspace=ws)
    o_ref, l_ref = OA.streaming_chunk_attention(bhld(q), oring, 2, bhld(k), bhld(v), w.W, False, w.scale)
    torch.cuda.synchronize()
    compare(O, LSE, o_ref, l_ref, what=f"after a caught key row, {splits} split(s)")
    assert sab.get_last_device_error() == 0


@needs_debug
def test_injected_workspace_tile_is_caught():
    """The split CTA whose partial tile would be the last one of the workspace
    is refused (the bound is lowered by one tile); only its query tile loses
    its merge, and the workspace stays usable."""
    w = synth.Workload("dbg_ws", B=1, H=2, D=128, Lc=256, R=2, W=2, seed=93)
    ring, oring, gen = _stream_ring(w, 2)
    q, k, v = synth.chunk_qkv(w, gen)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    splits = 3
    ws = ring.workspace(splits)
    O = torch.full_like(qd, 7.0)
    sab.debug_inject_bounds_error(sab.DEBUG_INJECT_WS_TILE)
    _, LSE = ring.attention(0, 2, qd, kd, vd, window=w.W, num_splits=splits, O=O, workspace=ws)
    assert sab.get_last_device_error() == sab.ERR_BOUNDS
    o_ref, l_ref = OA.streaming_chunk_attention(bhld(q), oring, 2, bhld(k), bhld(v), w.W, False, w.scale)
    torch.cuda.synchronize()
    # the refused tile is the last (b, h)'s last query tile: rows 128 .. 255 of head 1
    o = O.float().cpu().numpy()
    assert np.all(o[0, 128:, 1] == 7.0)
    compare(O[:, :, :1], LSE[:, :1], o_ref[:, :1], l_ref[:, :1], what="heads whose merge ran")
    compare(O[:, :128, 1:], LSE[:, 1:, :128], o_ref[:, 1:, :128], l_ref[:, 1:, :128], what="first tile of head 1")
    O, LSE = ring.attention(0, 2, qd, kd, vd, window=w.W, num_splits=splits, workspace=ws)
    torch.cuda.synchronize()
    compare(O, LSE, o_ref, l_ref, what="after a caught workspace tile")
    assert sab.get_last_device_error() == 0
