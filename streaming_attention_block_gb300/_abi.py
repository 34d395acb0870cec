"""ctypes marshalling for libsab.so.  Same names as the C ABI, without the
``sab_`` prefix.  Tensors are passed as device pointers taken from torch
tensors (which must be CUDA, contiguous and of the documented dtype); streams
default to torch's current stream."""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_INT8K_FP8V = 2

_STATUS = {
    0: "SAB_OK", 1: "SAB_ERR_INVALID_ARG", 2: "SAB_ERR_UNSUPPORTED", 3: "SAB_ERR_OUT_OF_RANGE",
    4: "SAB_ERR_WORKSPACE", 5: "SAB_ERR_CUDA", 6: "SAB_ERR_TIMEOUT", 7: "SAB_ERR_BOUNDS",
}
ERR_TIMEOUT = 6
ERR_BOUNDS = 7
# sab_debug_inject_bounds_error kinds
DEBUG_INJECT_APPEND_SLOT = 1
DEBUG_INJECT_KEY_ROW = 2
DEBUG_INJECT_WS_TILE = 3


class SabError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {_STATUS.get(self.status, self.status)}")


class RingDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "batch", "heads", "head_dim", "chunk_tokens", "ring_slots", "has_sink", "kv_dtype")]


_lib = None


def library_path() -> str:
    return os.environ.get("SAB_LIBRARY", os.path.join(_HERE, "libsab.so"))


def library() -> ctypes.CDLL:
    """Load libsab.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"libsab.so not found at {path}: build it with "
                          "`python -m streaming_attention_block_gb300.build` (there is no fallback)")
    lib = ctypes.CDLL(path)
    P, I, LL, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t, ctypes.c_float
    DP = ctypes.POINTER(RingDesc)
    sigs = {
        "sab_kv_ring_bytes": (SZ, [DP]),
        "sab_kv_ring_create": (I, [DP, P, SZ, P, ctypes.POINTER(P)]),
        "sab_kv_ring_destroy": (I, [P]),
        "sab_kv_ring_get_desc": (I, [P, DP]),
        "sab_kv_ring_layer_ptrs": (I, [P, I, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P),
                                       ctypes.POINTER(P)]),
        "sab_kv_ring_set_sink": (I, [P, I, P, P, P]),
        "sab_kv_ring_append": (I, [P, I, LL, P, P, P]),
        "sab_kv_ring_slot_of": (I, [P, I, LL, ctypes.POINTER(I)]),
        "sab_kv_ring_get_state": (I, [P, ctypes.POINTER(LL), ctypes.POINTER(I), ctypes.POINTER(I)]),
        "sab_kv_ring_set_state": (I, [P, ctypes.POINTER(LL), ctypes.POINTER(I), ctypes.POINTER(I)]),
        "sab_chunk_attention_workspace": (SZ, [P, I]),
        "sab_chunk_attention": (I, [P, I, LL, P, P, P, I, I, I, F, P, P, P, SZ, P]),
        "sab_chunk_attention_noalloc": (I, [P, I, LL, P, P, P, I, I, I, F, P, P, P]),
        "sab_chunk_attention_dev": (I, [P, I, P, P, P, P, I, I, I, F, P, P, P, SZ, P]),
        "sab_kv_ring_append_dev": (I, [P, I, P, P, P, P]),
        "sab_chunk_counter_add": (I, [P, LL, P]),
        "sab_block_causal_attention_workspace": (SZ, [I, I, I, I, I]),
        "sab_block_causal_attention": (I, [P, P, P, I, I, I, I, I, I, I, F, P, P, P, SZ, P]),
        "sab_get_last_device_error": (I, [P]),
        "sab_debug_bounds_enabled": (I, []),
        "sab_debug_inject_bounds_error": (I, [I]),
        "sab_selftest_bounded_wait": (I, [ctypes.c_ulonglong, P]),
        "sab_selftest_split_abort": (I, [P, I, LL, P, P, P, I, I, I, F, P, P, P, SZ, I, P]),
        "sab_qk_norm_rope": (I, [P, I, LL, P, P, P, P, P, P, P, P, P, I, P]),
        "sab_block_causal_attention_backward_workspace": (SZ, [I, I, I]),
        "sab_block_causal_attention_backward": (I, [P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, SZ, P]),
        "sab_memory_prefix_attention": (I, [P, P, P, I, I, I, I, I, P, I, I, F, P, P, P]),
        "sab_chunk_attention_fp8mma": (I, [P, I, LL, P, I, I, I, F, P, P, P, SZ, P]),
        "sab_memory_prefix_attention_backward": (I, [P, P, P, P, P, P, I, I, I, I, I, P, I, I, F, P, P, P, P, SZ,
                                                     P]),
        "sab_status_string": (ctypes.c_char_p, [I]),
        "sab_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise SabError(status, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor or a device pointer")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def status_string(status: int) -> str:
    return library().sab_status_string(int(status)).decode()


def version() -> str:
    return library().sab_version().decode()


def _desc(desc) -> RingDesc:
    if isinstance(desc, RingDesc):
        return desc
    return RingDesc(**desc)


def kv_ring_bytes(desc) -> int:
    return int(library().sab_kv_ring_bytes(ctypes.byref(_desc(desc))))


def kv_ring_create(desc, mem: torch.Tensor, stream=None) -> ctypes.c_void_p:
    d = _desc(desc)
    h = ctypes.c_void_p()
    _check(library().sab_kv_ring_create(ctypes.byref(d), _ptr(mem, torch.uint8, "mem"),
                                        mem.numel(), _stream(stream), ctypes.byref(h)), "kv_ring_create")
    return h


def kv_ring_destroy(handle):
    _check(library().sab_kv_ring_destroy(handle), "kv_ring_destroy")


def kv_ring_get_desc(handle) -> RingDesc:
    d = RingDesc()
    _check(library().sab_kv_ring_get_desc(handle, ctypes.byref(d)), "kv_ring_get_desc")
    return d


def kv_ring_layer_ptrs(handle, layer: int):
    k, v, ks, vs = (ctypes.c_void_p() for _ in range(4))
    _check(library().sab_kv_ring_layer_ptrs(handle, int(layer), ctypes.byref(k), ctypes.byref(v),
                                            ctypes.byref(ks), ctypes.byref(vs)), "kv_ring_layer_ptrs")
    return k.value, v.value, ks.value, vs.value


def kv_ring_set_sink(handle, layer: int, K, V, stream=None):
    _check(library().sab_kv_ring_set_sink(handle, int(layer), _ptr(K, torch.bfloat16, "K"),
                                          _ptr(V, torch.bfloat16, "V"), _stream(stream)), "kv_ring_set_sink")


def kv_ring_append(handle, layer: int, chunk: int, K, V, stream=None):
    _check(library().sab_kv_ring_append(handle, int(layer), int(chunk), _ptr(K, torch.bfloat16, "K"),
                                        _ptr(V, torch.bfloat16, "V"), _stream(stream)), "kv_ring_append")


def kv_ring_slot_of(handle, layer: int, chunk: int) -> int:
    s = ctypes.c_int()
    _check(library().sab_kv_ring_slot_of(handle, int(layer), int(chunk), ctypes.byref(s)), "kv_ring_slot_of")
    return s.value


def kv_ring_get_state(handle, num_layers: int):
    n = (ctypes.c_longlong * num_layers)()
    h = (ctypes.c_int * num_layers)()
    s = (ctypes.c_int * num_layers)()
    _check(library().sab_kv_ring_get_state(handle, n, h, s), "kv_ring_get_state")
    return list(n), list(h), list(s)


def kv_ring_set_state(handle, newest, held, sink_set):
    L = len(newest)
    _check(library().sab_kv_ring_set_state(handle, (ctypes.c_longlong * L)(*newest), (ctypes.c_int * L)(*held),
                                           (ctypes.c_int * L)(*sink_set)), "kv_ring_set_state")


def chunk_attention_workspace(handle, num_splits: int) -> int:
    return int(library().sab_chunk_attention_workspace(handle, int(num_splits)))


def chunk_attention(handle, layer: int, chunk: int, Q, K_cur, V_cur, window: int, use_sink: bool,
                    num_splits: int, softmax_scale: float, O, LSE=None, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().sab_chunk_attention(
        handle, int(layer), int(chunk), _ptr(Q, torch.bfloat16, "Q"), _ptr(K_cur, torch.bfloat16, "K_cur"),
        _ptr(V_cur, torch.bfloat16, "V_cur"), int(window), int(bool(use_sink)), int(num_splits),
        float(softmax_scale), _ptr(O, torch.bfloat16, "O"), _ptr(LSE, torch.float32, "LSE"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)), "chunk_attention")


def chunk_attention_noalloc(handle, layer: int, chunk: int, Q, K_cur, V_cur, window: int, use_sink: bool,
                            num_splits: int, softmax_scale: float, O, LSE=None, stream=None):
    """sab_chunk_attention_noalloc: the split merge uses the library's own
    device scratch instead of a caller workspace (see include/sab.h)."""
    _check(library().sab_chunk_attention_noalloc(
        handle, int(layer), int(chunk), _ptr(Q, torch.bfloat16, "Q"), _ptr(K_cur, torch.bfloat16, "K_cur"),
        _ptr(V_cur, torch.bfloat16, "V_cur"), int(window), int(bool(use_sink)), int(num_splits),
        float(softmax_scale), _ptr(O, torch.bfloat16, "O"), _ptr(LSE, torch.float32, "LSE"), _stream(stream)),
        "chunk_attention_noalloc")


def chunk_attention_dev(handle, layer: int, d_chunk, Q, K_cur, V_cur, window: int, use_sink: bool,
                        num_splits: int, softmax_scale: float, O, LSE=None, workspace=None, stream=None):
    """sab_chunk_attention_dev: the chunk index is read from ``d_chunk`` (a
    device int64 tensor) when the kernel runs, so the call can be captured
    once in a CUDA graph and replayed for every chunk (see include/sab.h)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().sab_chunk_attention_dev(
        handle, int(layer), _ptr(d_chunk, torch.int64, "d_chunk"), _ptr(Q, torch.bfloat16, "Q"),
        _ptr(K_cur, torch.bfloat16, "K_cur"), _ptr(V_cur, torch.bfloat16, "V_cur"), int(window),
        int(bool(use_sink)), int(num_splits), float(softmax_scale), _ptr(O, torch.bfloat16, "O"),
        _ptr(LSE, torch.float32, "LSE"), _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)),
        "chunk_attention_dev")


def kv_ring_append_dev(handle, layer: int, d_chunk, K, V, stream=None):
    """sab_kv_ring_append_dev: append into slot (*d_chunk mod R), chunk read on the device."""
    _check(library().sab_kv_ring_append_dev(handle, int(layer), _ptr(d_chunk, torch.int64, "d_chunk"),
                                            _ptr(K, torch.bfloat16, "K"), _ptr(V, torch.bfloat16, "V"),
                                            _stream(stream)), "kv_ring_append_dev")


def chunk_counter_add(d_chunk, delta: int = 1, stream=None):
    """sab_chunk_counter_add: *d_chunk += delta on the stream."""
    _check(library().sab_chunk_counter_add(_ptr(d_chunk, torch.int64, "d_chunk"), int(delta), _stream(stream)),
           "chunk_counter_add")


def block_causal_attention_backward_workspace(B: int, L: int, H: int) -> int:
    return int(library().sab_block_causal_attention_backward_workspace(B, L, H))


def block_causal_attention_backward(Q, K, V, O, dO, LSE, chunk_tokens: int, window: int, softmax_scale: float,
                                    dQ, dK, dV, workspace=None, stream=None):
    """sab_block_causal_attention_backward: (dQ, dK, dV) of block-causal
    attention from the forward's O and LSE (see include/sab.h)."""
    B, L, H, D = Q.shape
    if workspace is None:
        n = int(library().sab_block_causal_attention_backward_workspace(B, L, H))
        workspace = torch.empty(n, dtype=torch.uint8, device=Q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(library().sab_block_causal_attention_backward(
        _ptr(Q, torch.bfloat16, "Q"), _ptr(K, torch.bfloat16, "K"), _ptr(V, torch.bfloat16, "V"),
        _ptr(O, torch.bfloat16, "O"), _ptr(dO, torch.bfloat16, "dO"), _ptr(LSE, torch.float32, "LSE"),
        B, L, H, D, int(chunk_tokens), int(window), float(softmax_scale), _ptr(dQ, torch.bfloat16, "dQ"),
        _ptr(dK, torch.bfloat16, "dK"), _ptr(dV, torch.bfloat16, "dV"), _ptr(workspace, None, "workspace"),
        ws_bytes, _stream(stream)), "block_causal_attention_backward")


def chunk_attention_fp8mma(handle, layer: int, chunk: int, Q, window: int, use_sink: bool, softmax_scale: float,
                           O, LSE=None, stream=None, num_splits: int = 1, workspace=None):
    """sab_chunk_attention_fp8mma: chunk attention over an E4M3 ring with Q and
    P rounded to E4M3 for the tensor-core products (see include/sab.h);
    ``num_splits`` and ``workspace`` as in ``chunk_attention``."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().sab_chunk_attention_fp8mma(
        handle, int(layer), int(chunk), _ptr(Q, torch.bfloat16, "Q"), int(window), 1 if use_sink else 0,
        int(num_splits), float(softmax_scale), _ptr(O, torch.bfloat16, "O"), _ptr(LSE, torch.float32, "LSE"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)), "chunk_attention_fp8mma")


def memory_prefix_attention(Q, K, V, mem_pad: int, mem_len, chunk_tokens: int, window: int, softmax_scale: float,
                            O, LSE=None, stream=None):
    """sab_memory_prefix_attention: block-causal target chunks behind a
    per-sample memory prefix of mem_pad positions, mem_len (device int32 [B])
    of them real (see include/sab.h)."""
    B, L, H, D = Q.shape
    _check(library().sab_memory_prefix_attention(
        _ptr(Q, torch.bfloat16, "Q"), _ptr(K, torch.bfloat16, "K"), _ptr(V, torch.bfloat16, "V"),
        B, L, H, D, int(mem_pad), _ptr(mem_len, torch.int32, "mem_len"), int(chunk_tokens), int(window),
        float(softmax_scale), _ptr(O, torch.bfloat16, "O"), _ptr(LSE, torch.float32, "LSE"), _stream(stream)),
        "memory_prefix_attention")


def memory_prefix_attention_backward(Q, K, V, O, dO, LSE, mem_pad: int, mem_len, chunk_tokens: int, window: int,
                                     softmax_scale: float, dQ, dK, dV, workspace=None, stream=None):
    """sab_memory_prefix_attention_backward: (dQ, dK, dV) of
    memory_prefix_attention from its O and LSE (see include/sab.h)."""
    B, L, H, D = Q.shape
    if workspace is None:
        n = int(library().sab_block_causal_attention_backward_workspace(B, L, H))
        workspace = torch.empty(n, dtype=torch.uint8, device=Q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(library().sab_memory_prefix_attention_backward(
        _ptr(Q, torch.bfloat16, "Q"), _ptr(K, torch.bfloat16, "K"), _ptr(V, torch.bfloat16, "V"),
        _ptr(O, torch.bfloat16, "O"), _ptr(dO, torch.bfloat16, "dO"), _ptr(LSE, torch.float32, "LSE"),
        B, L, H, D, int(mem_pad), _ptr(mem_len, torch.int32, "mem_len"), int(chunk_tokens), int(window),
        float(softmax_scale), _ptr(dQ, torch.bfloat16, "dQ"), _ptr(dK, torch.bfloat16, "dK"),
        _ptr(dV, torch.bfloat16, "dV"), _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)),
        "memory_prefix_attention_backward")


def block_causal_attention_workspace(B: int, L: int, H: int, D: int, num_splits: int) -> int:
    return int(library().sab_block_causal_attention_workspace(B, L, H, D, num_splits))


def block_causal_attention(Q, K, V, chunk_tokens: int, window: int, num_splits: int, softmax_scale: float,
                           O, LSE=None, workspace=None, stream=None):
    B, L, H, D = Q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().sab_block_causal_attention(
        _ptr(Q, torch.bfloat16, "Q"), _ptr(K, torch.bfloat16, "K"), _ptr(V, torch.bfloat16, "V"),
        B, L, H, D, int(chunk_tokens), int(window), int(num_splits), float(softmax_scale),
        _ptr(O, torch.bfloat16, "O"), _ptr(LSE, torch.float32, "LSE"), _ptr(workspace, None, "workspace"),
        ws_bytes, _stream(stream)), "block_causal_attention")


def get_last_device_error(stream=None) -> int:
    return int(library().sab_get_last_device_error(_stream(stream)))


def debug_bounds_enabled() -> bool:
    """True when the loaded library is the debug build (device index checks)."""
    return bool(library().sab_debug_bounds_enabled())


def debug_inject_bounds_error(what: int):
    """sab_debug_inject_bounds_error (debug builds only)."""
    _check(library().sab_debug_inject_bounds_error(int(what)), "debug_inject_bounds_error")


# Canary bands: a device buffer can be allocated between two bands of
# GUARD_BYTE that no call may write.  While a watch is open every guarded
# allocation is recorded, and closing the watch counts the band bytes that
# changed (buffer overruns or underruns by any kernel that wrote near it).
GUARD_BYTE = 0xA5
_guard_watch = None


def _guarded(nbytes: int, guard: int, device, zero: bool = False):
    """(storage, view): ``view`` is ``nbytes`` of 256-byte-aligned device
    memory, with ``guard`` bytes (rounded up to 256) of canaries on each side."""
    g = (int(guard) + 255) // 256 * 256
    mem = torch.empty(nbytes + 2 * g + 256, dtype=torch.uint8, device=device)
    off = (-mem.data_ptr()) % 256 + g
    buf = mem[off:off + nbytes]
    if zero:
        buf.zero_()
    if g:
        mem[:off].fill_(GUARD_BYTE)
        mem[off + nbytes:].fill_(GUARD_BYTE)
        if _guard_watch is not None:
            _guard_watch.append((mem, ((0, off), (off + nbytes, mem.numel()))))
    return mem, buf


def guard_watch_begin():
    """Start recording guarded allocations."""
    global _guard_watch
    _guard_watch = []


def guard_watch_end() -> int:
    """Stop recording; return how many canary bytes of the recorded
    allocations no longer hold GUARD_BYTE (0: no call wrote outside them)."""
    global _guard_watch
    watched, _guard_watch = _guard_watch or [], None
    bad = 0
    for mem, bands in watched:
        for lo, hi in bands:
            bad += int((mem[lo:hi] != GUARD_BYTE).sum().item())
    return bad


def selftest_bounded_wait(timeout_ns: int, stream=None):
    """sab_selftest_bounded_wait: a device wait that nothing completes gives up
    after timeout_ns; read the result with get_last_device_error."""
    _check(library().sab_selftest_bounded_wait(int(timeout_ns), _stream(stream)), "selftest_bounded_wait")


def selftest_split_abort(handle, layer: int, chunk: int, Q, K_cur, V_cur, window: int, use_sink: bool,
                         num_splits: int, softmax_scale: float, O, LSE, workspace, abort_split: int, stream=None):
    """sab_selftest_split_abort: a split call (num_splits > 8, workspace merge)
    whose split ``abort_split`` reports itself as having given up a wait."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().sab_selftest_split_abort(
        handle, int(layer), int(chunk), _ptr(Q, torch.bfloat16, "Q"), _ptr(K_cur, torch.bfloat16, "K_cur"),
        _ptr(V_cur, torch.bfloat16, "V_cur"), int(window), int(bool(use_sink)), int(num_splits),
        float(softmax_scale), _ptr(O, torch.bfloat16, "O"), _ptr(LSE, torch.float32, "LSE"),
        _ptr(workspace, None, "workspace"), ws_bytes, int(abort_split), _stream(stream)), "selftest_split_abort")


class RopeDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("frames", "height", "width", "band_t", "band_h", "band_w")] + [
        ("base", ctypes.c_float), ("eps", ctypes.c_float)]


def qk_norm_rope(handle, layer: int, chunk: int, Q, K, V, rope: RopeDesc, Q_out, K_out=None, V_out=None,
                 gamma_q=None, gamma_k=None, append: bool = False, stream=None):
    """sab_qk_norm_rope: q' = RoPE(RMSNorm(q)), k' = RoPE(RMSNorm(k)) of one
    chunk, optionally appending k', v into the ring slot (see include/sab.h)."""
    _check(library().sab_qk_norm_rope(
        handle, int(layer), int(chunk), _ptr(Q, torch.bfloat16, "Q"), _ptr(K, torch.bfloat16, "K"),
        _ptr(V, torch.bfloat16, "V"), _ptr(gamma_q, torch.float32, "gamma_q"), _ptr(gamma_k, torch.float32, "gamma_k"),
        ctypes.byref(rope), _ptr(Q_out, torch.bfloat16, "Q_out"), _ptr(K_out, torch.bfloat16, "K_out"),
        _ptr(V_out, torch.bfloat16, "V_out"), int(bool(append)), _stream(stream)), "qk_norm_rope")


class KVRing:
    """A ring KV cache on torch-owned device memory (memory + handle).

    ``guard_bytes`` (default ``KVRing.default_guard_bytes``, 0) puts canary
    bands of that many bytes around the ring memory and around every
    workspace ``workspace()`` allocates (see ``guard_watch_begin``)."""

    default_guard_bytes = 0

    def __init__(self, num_layers, batch, heads, head_dim, chunk_tokens, ring_slots, has_sink=False,
                 kv_dtype=KV_BF16, device="cuda", stream=None, guard_bytes=None):
        self.desc = RingDesc(num_layers, batch, heads, head_dim, chunk_tokens, ring_slots, int(bool(has_sink)),
                             int(kv_dtype))
        nbytes = kv_ring_bytes(self.desc)
        if nbytes == 0:
            raise SabError(1, "invalid ring shape")
        self.guard_bytes = self.default_guard_bytes if guard_bytes is None else int(guard_bytes)
        self.mem, self.buf = _guarded(nbytes, self.guard_bytes, device)
        self.handle = kv_ring_create(self.desc, self.buf, stream)
        self.rows = (self.desc.has_sink + ring_slots) * chunk_tokens

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.sab_kv_ring_destroy(h)
            self.handle = None

    def _view(self, ptr, nbytes, dtype, shape):
        off = ptr - self.buf.data_ptr()
        return self.buf[off:off + nbytes].view(dtype).view(shape)

    def layer_views(self, layer):
        """(K, V, K_scale, V_scale) torch views of one layer's ring memory."""
        d = self.desc
        k, v, ks, vs = kv_ring_layer_ptrs(self.handle, layer)
        fp8 = d.kv_dtype != KV_BF16  # one byte per element (E4M3, or INT8 keys)
        dt, es = (torch.uint8, 1) if fp8 else (torch.bfloat16, 2)
        shape = (d.batch, d.heads, self.rows, d.head_dim)
        n = d.batch * d.heads * self.rows * d.head_dim * es
        K = self._view(k, n, dt, shape)
        V = self._view(v, n, dt, shape)
        if not fp8:
            return K, V, None, None
        sshape = (d.batch, d.heads, d.has_sink + d.ring_slots)
        sn = d.batch * d.heads * (d.has_sink + d.ring_slots) * 4
        return K, V, self._view(ks, sn, torch.float32, sshape), self._view(vs, sn, torch.float32, sshape)

    def set_sink(self, layer, K, V, stream=None):
        kv_ring_set_sink(self.handle, layer, K, V, stream)

    def append(self, layer, chunk, K, V, stream=None):
        kv_ring_append(self.handle, layer, chunk, K, V, stream)

    def slot_of(self, layer, chunk):
        return kv_ring_slot_of(self.handle, layer, chunk)

    def workspace(self, num_splits):
        n = chunk_attention_workspace(self.handle, num_splits)
        if n == 0:
            return None
        return _guarded(n, self.guard_bytes, self.buf.device, zero=True)[1]

    def attention(self, layer, chunk, Q, K_cur=None, V_cur=None, window=2, use_sink=False, num_splits=1,
                  softmax_scale=None, O=None, LSE=None, workspace=None, stream=None):
        d = self.desc
        if softmax_scale is None:
            softmax_scale = d.head_dim ** -0.5
        if O is None:
            O = torch.empty_like(Q)
        if LSE is None:
            LSE = torch.empty((d.batch, d.heads, d.chunk_tokens), dtype=torch.float32, device=Q.device)
        if num_splits > 1 and workspace is None:
            workspace = self.workspace(num_splits)
        chunk_attention(self.handle, layer, chunk, Q, K_cur, V_cur, window, use_sink, num_splits, softmax_scale,
                        O, LSE, workspace, stream)
        return O, LSE
