"""ctypes binding of the OSCAR C ABI (include/oscar.h).

Argument marshalling only: every function below calls the entry point of the
same name in ``liboscar_gb300.so`` and raises :class:`OscarError` on a
non-OK status.  There is no Python or CPU fallback; when the shared library is
missing or was built for another machine, loading fails loudly.
"""

import ctypes
import os
import threading

HEAD_DIM = 128
PAGE_TOKENS = 64
SINK_TOKENS = 64
RECENT_TOKENS = 256
GROUP = 64
MAX_GQA = 8
BLOCK_BYTES = 4608
NOALLOC_SCRATCH_BYTES = 16 << 20

OSCAR_OK = 0
STATUS_NAMES = {0: "OSCAR_OK", 1: "OSCAR_ERR_INVALID_ARG", 2: "OSCAR_ERR_UNSUPPORTED", 3: "OSCAR_ERR_NOT_LOADED",
                4: "OSCAR_ERR_CUDA", 5: "OSCAR_ERR_DEVICE_CHECK", 6: "OSCAR_ERR_WORKSPACE"}

OSCAR_DEVERR_PAGE = 1
OSCAR_DEVERR_SINK = 2
OSCAR_DEVERR_RING = 4
OSCAR_DEVERR_LENGTH = 8
OSCAR_DEVERR_TOKENS = 16
OSCAR_DEVERR_TIMEOUT = 32

OSCAR_APPEND_FRESH_RING = 1

OSCAR_ROT_U = 1
OSCAR_ROT_H = 2
OSCAR_ROT_P = 4
OSCAR_ROT_ALL = 7


class OscarError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s failed: %s" % (where, STATUS_NAMES.get(status, str(status))))


class oscar_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("sink", ctypes.c_int32),
                ("recent", ctypes.c_int32), ("group", ctypes.c_int32), ("device", ctypes.c_int32)]


class oscar_cache_view(ctypes.Structure):
    _fields_ = [("int2_pages", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("k_sink", ctypes.c_void_p), ("v_sink", ctypes.c_void_p), ("num_sink_pages", ctypes.c_int64),
                ("k_ring", ctypes.c_void_p), ("v_ring", ctypes.c_void_p), ("num_ring_slots", ctypes.c_int64),
                ("page_table", ctypes.c_void_p), ("max_pages_per_req", ctypes.c_int32),
                ("sink_page", ctypes.c_void_p), ("ring_slot", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("recent_page_table", ctypes.c_void_p)]


class oscar_append_args(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("n_tokens", ctypes.c_int32),
                ("max_tokens_per_req", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class oscar_decode_args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("out", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p),
                ("max_ctx_len", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


class oscar_bf16_cache_view(ctypes.Structure):
    _fields_ = [("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_table", ctypes.c_void_p), ("max_pages_per_req", ctypes.c_int32), ("batch", ctypes.c_int32)]


# name -> (restype, argtypes)
SIGNATURES = {
    "oscar_create": (ctypes.c_int, [ctypes.POINTER(oscar_config), ctypes.POINTER(ctypes.c_void_p)]),
    "oscar_destroy": (None, [ctypes.c_void_p]),
    "oscar_load_rotation": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_float, ctypes.c_float, ctypes.c_uint32]),
    "oscar_kv_append": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(oscar_cache_view),
                                       ctypes.POINTER(oscar_append_args), ctypes.c_void_p]),
    "oscar_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]),
    "oscar_decode_attention": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(oscar_cache_view),
                                              ctypes.POINTER(oscar_decode_args), ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_void_p]),
    "oscar_extend_attention": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(oscar_cache_view),
                                              ctypes.POINTER(oscar_decode_args), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_void_p]),
    "oscar_extend_workspace_bytes": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                        ctypes.c_int32]),
    "oscar_extend_chunk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(oscar_cache_view),
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_void_p]),
    "oscar_decode_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(oscar_cache_view),
                                         ctypes.POINTER(oscar_append_args), ctypes.POINTER(oscar_decode_args),
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "oscar_decode_attention_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(oscar_cache_view),
                                                      ctypes.POINTER(oscar_decode_args), ctypes.c_void_p]),
    "oscar_decode_attention_bf16": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(oscar_bf16_cache_view),
                                                   ctypes.POINTER(oscar_decode_args), ctypes.c_void_p,
                                                   ctypes.c_size_t, ctypes.c_void_p]),
    "oscar_calib_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64]),
    "oscar_calib_covariances": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                               ctypes.c_void_p]),
    "oscar_calib_clip_threshold": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                                  ctypes.c_uint32, ctypes.c_double, ctypes.POINTER(ctypes.c_double),
                                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "oscar_check_device_error": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "oscar_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]),
    "oscar_device_sm_count": (ctypes.c_int32, [ctypes.c_void_p]),
    "oscar_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None
_lock = threading.Lock()


def library_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboscar_gb300.so")


def load(build_if_missing=True):
    """Load (building first if needed) the shared library; raises if that is impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if build_if_missing:
            from . import build as _build
            try:
                path = _build.build()
            except RuntimeError:
                if not os.path.exists(path):
                    raise
        if not os.path.exists(path):
            raise RuntimeError("liboscar_gb300.so is missing: run int2_rotated_kv_oscar_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status, where):
    if status != OSCAR_OK:
        raise OscarError(status, where)


def _ptr(x):
    """Device/host address of a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def oscar_create(config):
    h = ctypes.c_void_p()
    _check(load().oscar_create(ctypes.byref(config), ctypes.byref(h)), "oscar_create")
    return h


def oscar_destroy(ctx):
    if ctx:
        load().oscar_destroy(ctx)


def oscar_load_rotation(ctx, layer, U_K, U_V, tau_k, tau_v, flags=OSCAR_ROT_ALL):
    """U_K, U_V: host float32 C-contiguous [128, 128] numpy arrays."""
    import numpy as np
    uk = np.ascontiguousarray(U_K, dtype=np.float32)
    uv = np.ascontiguousarray(U_V, dtype=np.float32)
    if uk.shape != (HEAD_DIM, HEAD_DIM) or uv.shape != (HEAD_DIM, HEAD_DIM):
        raise ValueError("U_K and U_V must be [128, 128]")
    _check(load().oscar_load_rotation(ctx, layer, uk.ctypes.data, uv.ctypes.data, float(tau_k), float(tau_v),
                                      flags), "oscar_load_rotation")


def oscar_kv_append(ctx, layer, view, args, stream=None):
    _check(load().oscar_kv_append(ctx, layer, ctypes.byref(view), ctypes.byref(args), _stream(stream)),
           "oscar_kv_append")


def oscar_decode_workspace_bytes(ctx, max_batch, max_ctx_len):
    return int(load().oscar_decode_workspace_bytes(ctx, max_batch, max_ctx_len))


def oscar_decode_attention(ctx, layer, view, args, workspace, workspace_bytes, stream=None):
    _check(load().oscar_decode_attention(ctx, layer, ctypes.byref(view), ctypes.byref(args), _ptr(workspace),
                                         workspace_bytes, _stream(stream)), "oscar_decode_attention")


def oscar_extend_attention(ctx, layer, view, args, limit, workspace, workspace_bytes, stream=None):
    """Decode-style attention of batch rows (a chunk's queries) with per-row causal limits (device int32)."""
    _check(load().oscar_extend_attention(ctx, layer, ctypes.byref(view), ctypes.byref(args), _ptr(limit),
                                         _ptr(workspace), workspace_bytes, _stream(stream)), "oscar_extend_attention")


def oscar_extend_workspace_bytes(ctx, batch, chunk, max_ctx_len):
    return int(load().oscar_extend_workspace_bytes(ctx, batch, chunk, max_ctx_len))


def oscar_extend_chunk(ctx, layer, view, q, out, ctx_len, pos0, chunk, max_ctx_len, workspace, workspace_bytes,
                       sm_scale=0.0, stream=None):
    """q bf16 [batch, chunk, Hq, 128], out fp32 (same), ctx_len and pos0 int32 [batch] (all device tensors)."""
    _check(load().oscar_extend_chunk(ctx, layer, ctypes.byref(view), _ptr(q), _ptr(out), _ptr(ctx_len), _ptr(pos0),
                                     chunk, max_ctx_len, float(sm_scale), _ptr(workspace), workspace_bytes,
                                     _stream(stream)), "oscar_extend_chunk")


def oscar_decode_step(ctx, layer, view, append, decode, workspace, workspace_bytes, stream=None):
    """Append one token per request, then decode, in one launch."""
    _check(load().oscar_decode_step(ctx, layer, ctypes.byref(view), ctypes.byref(append), ctypes.byref(decode),
                                    _ptr(workspace), workspace_bytes, _stream(stream)), "oscar_decode_step")


def oscar_decode_attention_noalloc(ctx, layer, view, args, stream=None):
    """Decode with the library's built-in scratch array instead of a caller workspace."""
    _check(load().oscar_decode_attention_noalloc(ctx, layer, ctypes.byref(view), ctypes.byref(args),
                                                 _stream(stream)), "oscar_decode_attention_noalloc")


def oscar_decode_attention_bf16(ctx, view, args, workspace, workspace_bytes, stream=None):
    _check(load().oscar_decode_attention_bf16(ctx, ctypes.byref(view), ctypes.byref(args), _ptr(workspace),
                                              workspace_bytes, _stream(stream)), "oscar_decode_attention_bf16")


def oscar_calib_workspace_bytes(n_queries, n_keys, n_kv_heads, n_clip_rows):
    return int(load().oscar_calib_workspace_bytes(n_queries, n_keys, n_kv_heads, n_clip_rows))


def oscar_calib_covariances(ctx, q, n_q, k, v, n_k, n_kv_heads, sm_scale, c_q, c_s, workspace, workspace_bytes,
                            stream=None):
    """q [n_q, 128], k and v [heads, n_k, 128] device float32; c_q, c_s device float64 [128, 128]."""
    _check(load().oscar_calib_covariances(ctx, _ptr(q), n_q, _ptr(k), _ptr(v), n_k, n_kv_heads, float(sm_scale),
                                          _ptr(c_q), _ptr(c_s), _ptr(workspace), workspace_bytes, _stream(stream)),
           "oscar_calib_covariances")


def oscar_calib_clip_threshold(ctx, x, n_rows, U, flags, percentile, workspace, workspace_bytes, stream=None):
    """x [n_rows, 128] device float32; U host float32 [128, 128]; returns the threshold (float)."""
    import numpy as np
    u = np.ascontiguousarray(U, dtype=np.float32)
    if u.shape != (HEAD_DIM, HEAD_DIM):
        raise ValueError("U must be [128, 128]")
    tau = ctypes.c_double(0.0)
    _check(load().oscar_calib_clip_threshold(ctx, _ptr(x), n_rows, u.ctypes.data, flags, float(percentile),
                                             ctypes.byref(tau), _ptr(workspace), workspace_bytes, _stream(stream)),
           "oscar_calib_clip_threshold")
    return float(tau.value)


def oscar_selftest_bounded_wait(ctx, polls, stream=None):
    """One bounded wait on a barrier nothing completes (sets OSCAR_DEVERR_TIMEOUT)."""
    _check(load().oscar_selftest_bounded_wait(ctx, int(polls), _stream(stream)), "oscar_selftest_bounded_wait")


def oscar_check_device_error(ctx, stream=None):
    """Returns the device error bits (0 when clean) after synchronising the stream."""
    bits = ctypes.c_uint32(0)
    st = load().oscar_check_device_error(ctx, _stream(stream), ctypes.byref(bits))
    if st not in (OSCAR_OK, 5):
        raise OscarError(st, "oscar_check_device_error")
    return int(bits.value)


def oscar_device_sm_count(ctx):
    return int(load().oscar_device_sm_count(ctx))


def oscar_status_string(status):
    return load().oscar_status_string(status).decode()
