"""Python binding of the C ABI in include/kvq.h (argument marshalling only).

Every step of the cache and of decode attention runs in the CUDA library
``_lib/libkvq.so``; this module only passes device pointers, sizes and the
CUDA stream.  If the library is missing it raises: there is no fallback.

Two layers:
  * functions named exactly like the C ABI (``kvq_create``, ``kvq_prefill_quantize``,
    ``kvq_append``, ``kvq_decode_attention``, ``kvq_destroy`` ...), taking raw
    integers (pointers, stream handles) or torch tensors;
  * ``KVCache``, a small owner object over one handle that takes torch tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

# KVQ_LIB selects another build of the library (the debug build of the tests)
LIB_PATH = os.environ.get("KVQ_LIB") or _build.LIB

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = -1
KVQ_ERR_UNSUPPORTED = -2
KVQ_ERR_CAPACITY = -3
KVQ_ERR_STATE = -4
KVQ_ERR_CUDA = -5
KVQ_ERR_OOM = -6


class KVQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class kvq_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_tokens", ctypes.c_int64), ("k_bits", ctypes.c_int32),
                ("v_bits", ctypes.c_int32), ("group_size", ctypes.c_int32), ("residual", ctypes.c_int32),
                ("k_sparse", ctypes.c_int32), ("rope", ctypes.c_int32), ("rope_base", ctypes.c_float),
                ("softmax_scale", ctypes.c_float), ("sink_tokens", ctypes.c_int32), ("codebook", ctypes.c_int32)]


class kvq_unit_view(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("kcodes", "kz", "ks", "vcodes", "vz", "vs", "sp_idx", "sp_val",
                                               "wk", "wv")] + \
               [(n, ctypes.c_int64) for n in ("kcodes_bytes", "kmeta_bytes", "vcodes_bytes", "vmeta_bytes",
                                              "sp_idx_bytes", "sp_val_bytes", "window_bytes")] + \
               [("sk", ctypes.c_void_p), ("sv", ctypes.c_void_p), ("sink_bytes", ctypes.c_int64)]


class kvq_page_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("page_bytes", "kcodes_offset", "kmeta_offset", "vcodes_offset",
                                              "vmeta_offset", "sp_idx_offset", "sp_val_offset")] + \
               [("tokens_per_page", ctypes.c_int32), ("fragment_order", ctypes.c_int32)]


_P = ctypes.c_void_p
_lock = threading.Lock()
_lib = None

# every symbol include/kvq.h declares, with (restype, argtypes)
SIGNATURES = {
    "kvq_create": (ctypes.c_int, [ctypes.POINTER(kvq_config), ctypes.c_int, ctypes.POINTER(_P)]),
    "kvq_destroy": (ctypes.c_int, [_P]),
    "kvq_prefill_quantize": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, _P]),
    "kvq_append": (ctypes.c_int, [_P, _P, _P, _P]),
    "kvq_decode_attention": (ctypes.c_int, [_P, _P, _P, _P]),
    "kvq_decode_step": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "kvq_reset": (ctypes.c_int, [_P]),
    "kvq_set_codebooks": (ctypes.c_int, [_P, _P, _P]),
    "kvq_decode_attention_noalloc": (ctypes.c_int, [ctypes.POINTER(kvq_config), _P, ctypes.c_int64, _P, _P,
                                                    ctypes.c_int64, _P, _P, _P]),
    "kvq_noalloc_sync_status": (ctypes.c_int, [_P]),
    "kvq_get_state": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_int32)]),
    "kvq_unit_sizes": (ctypes.c_int, [_P, ctypes.POINTER(kvq_unit_view)]),
    "kvq_export_unit": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(kvq_unit_view), _P]),
    "kvq_set_splits": (ctypes.c_int, [_P, ctypes.c_int32]),
    "kvq_get_splits": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "kvq_sync_status": (ctypes.c_int, [_P, _P]),
    "kvq_test_inject": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64]),
    "kvq_debug_check": (ctypes.c_int, [_P]),
    "kvq_set_device_allocator": (ctypes.c_int, [_P, _P, _P]),
    "kvq_launch_count": (ctypes.c_int64, [_P]),
    "kvq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvq_version": (ctypes.c_int32, []),
    "kvq_page_layout": (ctypes.c_int, [ctypes.POINTER(kvq_config), ctypes.POINTER(kvq_page_info)]),
    "kvq_axis_quantize": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]),
    "kvq_axis_dequantize": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, _P, _P]),
    "kvq_axis_attention": (ctypes.c_int, [_P, _P, ctypes.c_int32, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,
                                          ctypes.c_int32, ctypes.c_float, _P, _P, _P]),
}

KVQ_AXIS_TOKENS = 0    # groups of G tokens of one channel (per-channel scales)
KVQ_AXIS_CHANNELS = 1  # groups of G channels of one token (per-token scales)


def lib():
    """Load libkvq.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                                   f"g.build()'` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().kvq_status_string(status).decode()
    except RuntimeError:
        return "library not loaded"


def _check(status: int, what: str):
    if status != KVQ_OK:
        raise KVQError(status, what)


def _ptr(x):
    """Device pointer of a torch tensor, or an integer address as given."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream, device=None):
    if stream is None:
        import torch
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(batch, num_kv_heads, num_q_heads, head_dim, max_tokens, k_bits, v_bits, group_size, residual,
                k_sparse=0, rope=0, rope_base=10000.0, softmax_scale=None, sink_tokens=0, codebook=0) -> kvq_config:
    if softmax_scale is None:
        softmax_scale = 1.0 / float(head_dim) ** 0.5
    return kvq_config(batch, num_kv_heads, num_q_heads, head_dim, max_tokens, k_bits, v_bits, group_size, residual,
                      k_sparse, rope, rope_base, softmax_scale, sink_tokens, codebook)


# ------------------------------------------------------------------ C-ABI named functions

def kvq_create(cfg: kvq_config, device: int = 0) -> int:
    h = _P()
    _check(lib().kvq_create(ctypes.byref(cfg), device, ctypes.byref(h)), "kvq_create")
    return h.value


def kvq_page_layout(cfg: kvq_config) -> dict:
    """Byte layout of one page of a configuration (host arithmetic, no GPU needed)."""
    info = kvq_page_info()
    _check(lib().kvq_page_layout(ctypes.byref(cfg), ctypes.byref(info)), "kvq_page_layout")
    return {n: getattr(info, n) for n, _ in kvq_page_info._fields_}


def kvq_destroy(handle) -> None:
    _check(lib().kvq_destroy(handle), "kvq_destroy")


def kvq_prefill_quantize(handle, k, v, n_tokens: int, stream=None) -> None:
    _check(lib().kvq_prefill_quantize(handle, _ptr(k), _ptr(v), n_tokens, _stream(stream)), "kvq_prefill_quantize")


def kvq_append(handle, k, v, stream=None) -> None:
    _check(lib().kvq_append(handle, _ptr(k), _ptr(v), _stream(stream)), "kvq_append")


def kvq_decode_attention(handle, q, out, stream=None) -> None:
    _check(lib().kvq_decode_attention(handle, _ptr(q), _ptr(out), _stream(stream)), "kvq_decode_attention")


def kvq_decode_step(handle, k, v, q, out, stream=None) -> None:
    _check(lib().kvq_decode_step(handle, _ptr(k), _ptr(v), _ptr(q), _ptr(out), _stream(stream)), "kvq_decode_step")


def kvq_decode_attention_noalloc(cfg: kvq_config, pages, pages_per_unit: int, window_k, window_v, n_tokens: int,
                                 q, out, stream=None) -> None:
    """Decode attention over caller-owned packed buffers, with no device allocation (see include/kvq.h)."""
    _check(lib().kvq_decode_attention_noalloc(ctypes.byref(cfg), _ptr(pages), pages_per_unit, _ptr(window_k),
                                              _ptr(window_v), n_tokens, _ptr(q), _ptr(out), _stream(stream)),
           "kvq_decode_attention_noalloc")


def kvq_noalloc_sync_status(stream=None) -> int:
    """Status of kvq_decode_attention_noalloc on the current device (clears a recorded error)."""
    return int(lib().kvq_noalloc_sync_status(_stream(stream)))


def kvq_reset(handle) -> None:
    _check(lib().kvq_reset(handle), "kvq_reset")


def kvq_get_state(handle):
    t, tq, nr = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    _check(lib().kvq_get_state(handle, ctypes.byref(t), ctypes.byref(tq), ctypes.byref(nr)), "kvq_get_state")
    return t.value, tq.value, nr.value


def kvq_set_splits(handle, splits: int) -> None:
    _check(lib().kvq_set_splits(handle, splits), "kvq_set_splits")


def kvq_get_splits(handle) -> int:
    s = ctypes.c_int32()
    _check(lib().kvq_get_splits(handle, ctypes.byref(s)), "kvq_get_splits")
    return s.value


def kvq_sync_status(handle, stream=None) -> int:
    return int(lib().kvq_sync_status(handle, _stream(stream)))


def kvq_test_inject(handle, withhold_page: int, wait_limit_ns: int) -> None:
    """Test hook: shorten the decode kernels' wait limit and leave one page uncopied (see include/kvq.h)."""
    _check(lib().kvq_test_inject(handle, withhold_page, wait_limit_ns), "kvq_test_inject")


def kvq_debug_check(handle) -> int:
    """Debug builds: error word and buffer canaries of a cache (KVQ_OK when intact)."""
    return int(lib().kvq_debug_check(handle))


# C function types of kvq_set_device_allocator
KVQ_ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p)
KVQ_FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p)


def kvq_set_device_allocator(alloc=None, free_fn=None, user=None) -> None:
    """Device allocator of caches created from now on: KVQ_ALLOC_FN / KVQ_FREE_FN objects (keep them
    alive while any cache made with them exists), or None and None for cudaMalloc / cudaFree."""
    _check(lib().kvq_set_device_allocator(ctypes.cast(alloc, ctypes.c_void_p) if alloc else None,
                                          ctypes.cast(free_fn, ctypes.c_void_p) if free_fn else None, user),
           "kvq_set_device_allocator")


def kvq_launch_count(handle) -> int:
    return int(lib().kvq_launch_count(handle))


def kvq_export_unit(handle, b: int, kvh: int, cfg: kvq_config, stream=None) -> dict:
    """Unit (b, kvh) in the canonical host layout (numpy arrays), waiting for `stream`."""
    sizes = kvq_unit_view()
    _check(lib().kvq_unit_sizes(handle, ctypes.byref(sizes)), "kvq_unit_sizes")
    t, tq, nr = kvq_get_state(handle)
    ns = t - tq - nr
    D, G, nsp = cfg.head_dim, cfg.group_size, cfg.k_sparse
    out = dict(
        kcodes=np.zeros((tq, D * cfg.k_bits // 32), np.uint32), kz=np.zeros((tq // G, D), np.uint16),
        ks=np.zeros((tq // G, D), np.uint16), vcodes=np.zeros((tq, D * cfg.v_bits // 32), np.uint32),
        vz=np.zeros((tq, D // G), np.uint16), vs=np.zeros((tq, D // G), np.uint16),
        sp_idx=np.zeros((tq, nsp), np.uint8), sp_val=np.zeros((tq, nsp), np.uint16),
        wk=np.zeros((nr, D), np.uint16), wv=np.zeros((nr, D), np.uint16))
    sink = dict(sk=np.zeros((ns, D), np.uint16), sv=np.zeros((ns, D), np.uint16))
    assert out["kcodes"].nbytes == sizes.kcodes_bytes and out["wk"].nbytes == sizes.window_bytes
    assert sink["sk"].nbytes == sizes.sink_bytes
    ptr = lambda a: a.ctypes.data if a.size else None  # noqa: E731
    view = kvq_unit_view(*[ptr(a) for a in out.values()], *[0] * 7, ptr(sink["sk"]), ptr(sink["sv"]), 0)
    out.update(sink)
    _check(lib().kvq_export_unit(handle, b, kvh, ctypes.byref(view), _stream(stream)), "kvq_export_unit")
    return out


def kvq_set_codebooks(handle, k_levels, v_levels) -> None:
    """Non-uniform levels (in steps) of a codebook cache: host sequences of 2^k_bits and 2^v_bits floats."""
    k = np.ascontiguousarray(k_levels, dtype=np.float32)
    v = np.ascontiguousarray(v_levels, dtype=np.float32)
    _check(lib().kvq_set_codebooks(handle, k.ctypes.data, v.ctypes.data), "kvq_set_codebooks")


def kvq_axis_quantize(x, n_units, n_tokens, head_dim, bits, group_size, axis, codes, zero, scale, stream=None):
    _check(lib().kvq_axis_quantize(_ptr(x), n_units, n_tokens, head_dim, bits, group_size, axis, _ptr(codes),
                                   _ptr(zero), _ptr(scale), _stream(stream)), "kvq_axis_quantize")


def kvq_axis_dequantize(codes, zero, scale, n_units, n_tokens, head_dim, group_size, axis, out, stream=None):
    _check(lib().kvq_axis_dequantize(_ptr(codes), _ptr(zero), _ptr(scale), n_units, n_tokens, head_dim, group_size,
                                     axis, _ptr(out), _stream(stream)), "kvq_axis_dequantize")


def kvq_axis_attention(k, v, kv_f32, q, n_units, heads_per_unit, n_tokens, head_dim, softmax_scale, scores, out,
                       stream=None):
    _check(lib().kvq_axis_attention(_ptr(k), _ptr(v), kv_f32, _ptr(q), n_units, heads_per_unit, n_tokens, head_dim,
                                    softmax_scale, _ptr(scores), _ptr(out), _stream(stream)), "kvq_axis_attention")


# ------------------------------------------------------------------ owner object

class KVCache:
    """One layer's quantized KV cache on one GPU (torch tensors in, torch tensors out)."""

    def __init__(self, batch, num_kv_heads, num_q_heads, head_dim, max_tokens, k_bits=2, v_bits=2, group_size=32,
                 residual=128, k_sparse=0, rope=0, rope_base=10000.0, softmax_scale=None, device=0, sink_tokens=0,
                 k_levels=None, v_levels=None):
        self.cfg = make_config(batch, num_kv_heads, num_q_heads, head_dim, max_tokens, k_bits, v_bits, group_size,
                               residual, k_sparse, rope, rope_base, softmax_scale, sink_tokens,
                               0 if k_levels is None else 1)
        self.device = device
        self.handle = kvq_create(self.cfg, device)
        if k_levels is not None:
            kvq_set_codebooks(self.handle, k_levels, v_levels)

    @classmethod
    def for_workload(cls, w, device=0, max_tokens=None):
        return cls(w.batch, w.kv_heads, w.q_heads, w.head_dim, max_tokens or w.max_tokens, w.k_bits, w.v_bits,
                   w.group, w.residual, w.k_sparse, w.rope, w.rope_base, w.softmax_scale, device,
                   getattr(w, "sink", 0), getattr(w, "k_levels", None) or None, getattr(w, "v_levels", None) or None)

    def _need(self, t, shape, name):
        import torch
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
        if not t.is_cuda or t.dtype != torch.float16 or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: need a contiguous CUDA fp16 tensor of shape {tuple(shape)}, got "
                             f"{t.device} {t.dtype} {tuple(t.shape)} contiguous={t.is_contiguous()}")

    def prefill_quantize(self, k, v, stream=None):
        c = self.cfg
        n = k.shape[2]
        self._need(k, (c.batch, c.num_kv_heads, n, c.head_dim), "k")
        self._need(v, (c.batch, c.num_kv_heads, n, c.head_dim), "v")
        kvq_prefill_quantize(self.handle, k, v, n, _stream(stream, self.device))

    def append(self, k, v, stream=None):
        c = self.cfg
        self._need(k, (c.batch, c.num_kv_heads, c.head_dim), "k")
        self._need(v, (c.batch, c.num_kv_heads, c.head_dim), "v")
        kvq_append(self.handle, k, v, _stream(stream, self.device))

    def decode_attention(self, q, out=None, stream=None):
        import torch
        c = self.cfg
        self._need(q, (c.batch, c.num_q_heads, c.head_dim), "q")
        if out is None:
            out = torch.empty_like(q)
        self._need(out, (c.batch, c.num_q_heads, c.head_dim), "out")
        kvq_decode_attention(self.handle, q, out, _stream(stream, self.device))
        return out

    def decode_step(self, k, v, q, out=None, stream=None):
        """append(k, v) then decode_attention(q) in one call (one launch, two on a flush)."""
        import torch
        c = self.cfg
        self._need(k, (c.batch, c.num_kv_heads, c.head_dim), "k")
        self._need(v, (c.batch, c.num_kv_heads, c.head_dim), "v")
        self._need(q, (c.batch, c.num_q_heads, c.head_dim), "q")
        if out is None:
            out = torch.empty_like(q)
        self._need(out, (c.batch, c.num_q_heads, c.head_dim), "out")
        kvq_decode_step(self.handle, k, v, q, out, _stream(stream, self.device))
        return out

    def reset(self):
        kvq_reset(self.handle)

    def state(self):
        return kvq_get_state(self.handle)

    def export_unit(self, b, kvh, stream=None):
        return kvq_export_unit(self.handle, b, kvh, self.cfg, _stream(stream, self.device))

    def set_splits(self, n):
        kvq_set_splits(self.handle, n)

    def splits(self):
        return kvq_get_splits(self.handle)

    def sync_status(self, stream=None):
        return kvq_sync_status(self.handle, _stream(stream, self.device))

    def launch_count(self):
        return kvq_launch_count(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            kvq_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
