"""CPU checks of the C-ABI library: it loads, exports every symbol that
include/sab.h declares, and its pure-host entry points (sizes, validation that
fails before any CUDA call, status strings) behave as documented."""

import ctypes
import os
import re

import pytest

import streaming_attention_block_gb300 as sab

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "sab.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sab_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from streaming_attention_block_gb300.build import build
    build()
    return sab.library()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("sab_kv_ring_create", "sab_kv_ring_append", "sab_chunk_attention", "sab_block_causal_attention"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert sab.status_string(0) == "SAB_OK"
    assert sab.status_string(6) == "SAB_ERR_TIMEOUT"
    assert sab.status_string(7) == "SAB_ERR_BOUNDS"
    assert "sm_103a" in sab.version()


def test_release_build_has_no_index_checks(lib):
    assert not sab.debug_bounds_enabled()
    # the injection hook exists in every build but is refused outside a debug build
    assert lib.sab_debug_inject_bounds_error(sab.DEBUG_INJECT_APPEND_SLOT) == 2  # SAB_ERR_UNSUPPORTED


def test_debug_build_exports_the_same_boundary_with_checks_on():
    """libsab_debug.so (-DSAB_DEBUG_BOUNDS): same exports; the checks are on and
    the injection hook validates its argument (host-only calls, no GPU)."""
    from streaming_attention_block_gb300.build import DEBUG_LIB, build
    build(debug_bounds=True)
    dl = ctypes.CDLL(DEBUG_LIB)
    for name in _declared():
        assert hasattr(dl, name), name
    dl.sab_debug_inject_bounds_error.argtypes = [ctypes.c_int]
    assert dl.sab_debug_bounds_enabled() == 1
    assert dl.sab_debug_inject_bounds_error(99) == 1   # SAB_ERR_INVALID_ARG
    assert dl.sab_debug_inject_bounds_error(-1) == 1
    assert dl.sab_debug_inject_bounds_error(sab.DEBUG_INJECT_WS_TILE) == 0
    assert dl.sab_debug_inject_bounds_error(0) == 0    # cancels it


def test_ring_bytes(lib):
    d = dict(num_layers=30, batch=1, heads=12, head_dim=128, chunk_tokens=1536, ring_slots=2, has_sink=0,
             kv_dtype=sab.KV_BF16)
    per = 12 * 2 * 1536 * 128 * 2
    assert sab.kv_ring_bytes(d) == 30 * 2 * per
    d8 = dict(d, kv_dtype=sab.KV_FP8_E4M3, has_sink=1, ring_slots=20, chunk_tokens=405, heads=24, num_layers=1)
    codes = 24 * 21 * 405 * 128
    codes_al = (codes + 255) // 256 * 256
    scales_al = (24 * 21 * 4 + 255) // 256 * 256
    assert sab.kv_ring_bytes(d8) == 2 * codes_al + 2 * scales_al
    # INT8 keys / E4M3 values: the same byte layout
    assert sab.kv_ring_bytes(dict(d8, kv_dtype=sab.KV_INT8K_FP8V)) == 2 * codes_al + 2 * scales_al
    for bad in (dict(d, head_dim=96), dict(d, ring_slots=0), dict(d, kv_dtype=7), dict(d, has_sink=2)):
        assert sab.kv_ring_bytes(bad) == 0


def test_workspace_sizes(lib):
    assert sab.block_causal_attention_workspace(2, 30720, 12, 128, 1) == 0
    n = sab.block_causal_attention_workspace(1, 405, 24, 128, 8)
    # 405 rows -> 4 query tiles of 128 -> 512 padded rows; one counter per (b, h, tile)
    cnt = (24 * 4 * 4 + 255) // 256 * 256
    o = (8 * 24 * 512 * 128 * 4 + 255) // 256 * 256
    lse = (8 * 24 * 512 * 4 + 255) // 256 * 256
    assert n == cnt + o + lse
    assert sab.block_causal_attention_workspace(1, 405, 24, 96, 8) == 0
    assert lib.sab_chunk_attention_workspace(None, 8) == 0


def test_validation_before_any_cuda_call(lib):
    d = sab.RingDesc(1, 1, 2, 64, 32, 2, 0, 0)
    h = ctypes.c_void_p()
    assert lib.sab_kv_ring_create(ctypes.byref(d), None, 1 << 20, None, ctypes.byref(h)) == 1
    assert lib.sab_kv_ring_create(ctypes.byref(d), ctypes.c_void_p(256), 16, None, ctypes.byref(h)) == 1
    assert lib.sab_kv_ring_append(None, 0, 0, ctypes.c_void_p(256), ctypes.c_void_p(256), None) == 1
    assert lib.sab_chunk_attention(None, 0, 0, None, None, None, 2, 0, 1, 0.1, None, None, None, 0, None) == 1
    assert lib.sab_block_causal_attention(None, None, None, 1, 1, 1, 64, 1, 1, 1, 0.1, None, None, None, 0,
                                          None) == 1
    p = ctypes.c_void_p(4096)
    assert lib.sab_block_causal_attention(p, p, p, 1, 128, 1, 96, 64, 1, 1, 0.1, p, None, None, 0, None) == 1
    assert lib.sab_block_causal_attention(p, p, p, 1, 128, 1, 64, 64, -1, 1, 0.1, p, None, None, 0, None) == 1
    # graph-mode entry points: null / misaligned device chunk index, no ring
    assert lib.sab_chunk_attention_dev(None, 0, None, p, None, None, 2, 0, 1, 0.1, p, None, None, 0, None) == 1
    assert lib.sab_chunk_attention_dev(None, 0, ctypes.c_void_p(4100), p, None, None, 2, 0, 1, 0.1, p, None, None,
                                       0, None) == 1
    assert lib.sab_kv_ring_append_dev(None, 0, p, p, p, None) == 1
    assert lib.sab_chunk_counter_add(None, 1, None) == 1
    assert lib.sab_chunk_counter_add(ctypes.c_void_p(4100), 1, None) == 1
    assert lib.sab_selftest_bounded_wait(10, None) == 1  # limit outside 1 ms .. 2 s
    # E4M3-product entry: no ring
    assert lib.sab_chunk_attention_fp8mma(None, 0, 0, p, 2, 0, 1, 0.1, p, None, None, 0, None) == 1
    assert lib.sab_kv_ring_destroy(None) == 0


def test_memory_prefix_validation_before_any_cuda_call(lib):
    p = ctypes.c_void_p(256)  # aligned dummy: validation fails before it is used
    args = lambda M, ml: (p, p, p, 2, 512, 2, 128, M, ml, 128, 2, 0.1, p, None, None)
    assert lib.sab_memory_prefix_attention(*args(513, p)) == 1    # mem_pad > L
    assert lib.sab_memory_prefix_attention(*args(-1, p)) == 1     # negative
    assert lib.sab_memory_prefix_attention(*args(64, None)) == 1  # lengths missing
    assert lib.sab_memory_prefix_attention(*args(64, ctypes.c_void_p(258))) == 1  # misaligned lengths
    bw = lambda M, ml: (p, p, p, p, p, p, 2, 512, 2, 128, M, ml, 128, 2, 0.1, p, p, p, p, 1 << 20, None)
    assert lib.sab_memory_prefix_attention_backward(*bw(600, p)) == 1
    assert lib.sab_memory_prefix_attention_backward(*bw(64, None)) == 1
