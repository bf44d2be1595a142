"""Thin Python binding of libevict (argument marshalling only).

Functions carry the C names of include/evict.h and take raw device pointers
(ints) and sizes; every step of the eviction path runs in the library's
CUDA kernels. ``EvictCache`` is a convenience wrapper that takes torch
tensors, passes their ``data_ptr()`` and the current CUDA stream, and wraps
the returned view as zero-copy torch tensors.

There is no fallback: if libevict.so is missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libevict.so")

EVICT_OK, EVICT_EINVAL, EVICT_ELIMIT, EVICT_ECUDA, EVICT_EDEVICE, EVICT_ENUM = range(6)
EVICT_KNORM, EVICT_QFILTERS, EVICT_CURDKV, EVICT_H2O = range(4)
EVICT_BF16, EVICT_FP32 = range(2)
HEAD_DIM = 128
MAX_GROUP = 32
METHODS = {"knorm": EVICT_KNORM, "qfilters": EVICT_QFILTERS, "curdkv": EVICT_CURDKV, "h2o": EVICT_H2O}
DTYPES = {"bf16": EVICT_BF16, "fp32": EVICT_FP32}


class EvictConfig(ctypes.Structure):
    _fields_ = [
        ("method", ctypes.c_int), ("dtype", ctypes.c_int), ("batch", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("budget", ctypes.c_int),
        ("n_sink", ctypes.c_int), ("recent", ctypes.c_int), ("max_block", ctypes.c_int),
        ("max_kept", ctypes.c_int), ("keep_low", ctypes.c_int), ("sign", ctypes.c_int),
        ("filters", ctypes.c_void_p), ("n_filter_heads", ctypes.c_int), ("rank_cap", ctypes.c_int),
        ("stream", ctypes.c_void_p), ("calib_tokens", ctypes.c_int), ("per_token", ctypes.c_int),
    ]


class EvictView(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("score", ctypes.c_void_p), ("n_kept", ctypes.c_int32), ("capacity", ctypes.c_int32)]


class EvictStats(ctypes.Structure):
    _fields_ = [("tokens_seen", ctypes.c_int64), ("tokens_kept", ctypes.c_int64),
                ("kept_bytes", ctypes.c_int64), ("full_seq_bytes", ctypes.c_int64),
                ("compression_ratio", ctypes.c_double), ("offset", ctypes.c_int64)]


class EvictKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class EvictError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libevict error {code}: {msg}")
        self.code = code


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGNATURES = {
    "evict_init": (_I, [ctypes.POINTER(EvictConfig), ctypes.POINTER(_P)]),
    "evict_update_and_fetch": (_I, [_P, _P, _P, _P, _I, ctypes.POINTER(EvictView)]),
    "evict_update_and_fetch_group": (_I, [ctypes.POINTER(_P), _I, ctypes.POINTER(_P), ctypes.POINTER(_P),
                                          ctypes.POINTER(_P), _I, ctypes.POINTER(EvictView)]),
    "evict_update_and_fetch_host": (_I, [_P, _P, _P, _P, _I, ctypes.POINTER(EvictView)]),
    "evict_get_view": (_I, [_P, ctypes.POINTER(EvictView)]),
    "evict_stats": (_I, [_P, ctypes.POINTER(EvictStats)]),
    "evict_set_state": (_I, [_P, _P, _P, _P, _P, _I, ctypes.c_int64]),
    "evict_reset": (_I, [_P]),
    "evict_set_stream": (_I, [_P, _P]),
    "evict_sync": (_I, [_P]),
    "evict_destroy": (None, [_P]),
    "evict_qfilters_calibrate": (_I, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "evict_set_profiling": (_I, [_P, _I]),
    "evict_kernel_times": (_I, [_P, ctypes.POINTER(EvictKernelTime), _I, ctypes.POINTER(_I)]),
    "evict_compaction_rows": (_I, [_P, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "evict_prefill_noalloc": (_I, [ctypes.POINTER(EvictConfig), _P, _P, _P, _I, _P, _P, _P, _P]),
    "evict_noalloc_status": (_I, [_P]),
    "evict_curdkv_scores": (_I, [_P, _P, _P, ctypes.POINTER(_I)]),
    "evict_qfilters_filters": (_I, [_P, _P, ctypes.POINTER(_I)]),
    "evict_launch_count": (ctypes.c_int64, []),
    "evict_last_error": (ctypes.c_char_p, []),
}


def load(path: str = LIB_PATH):
    """Load libevict.so (once). Raises OSError if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: build it with __graft_entry__.build() (there is no CPU fallback)")
    try:
        import torch  # noqa: F401  (loads the CUDA runtime first so both share it)
    except ImportError:
        pass
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(code: int):
    if code != EVICT_OK:
        msg = load().evict_last_error().decode(errors="replace")
        raise EvictError(code, msg)


# --------------------------------------------------------------------------
# Plain C-name wrappers (pointers as ints)
# --------------------------------------------------------------------------
def evict_init(cfg: EvictConfig) -> int:
    h = _P()
    check(load().evict_init(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def evict_update_and_fetch(h, k_ptr, v_ptr, pos_ptr, m) -> EvictView:
    view = EvictView()
    check(load().evict_update_and_fetch(h, k_ptr, v_ptr, pos_ptr, m, ctypes.byref(view)))
    return view


def evict_update_and_fetch_group(handles, k_ptrs, v_ptrs, pos_ptrs, m):
    n = len(handles)
    arr = lambda xs: (_P * n)(*[x if x else None for x in xs])
    views = (EvictView * n)()
    pos_arr = arr(pos_ptrs) if pos_ptrs is not None else None
    check(load().evict_update_and_fetch_group(arr(handles), n, arr(k_ptrs), arr(v_ptrs), pos_arr, m, views))
    return list(views)


def evict_update_and_fetch_host(h, k_host_ptr, v_host_ptr, pos_host_ptr, m) -> EvictView:
    view = EvictView()
    check(load().evict_update_and_fetch_host(h, k_host_ptr, v_host_ptr, pos_host_ptr, m, ctypes.byref(view)))
    return view


def evict_get_view(h) -> EvictView:
    view = EvictView()
    check(load().evict_get_view(h, ctypes.byref(view)))
    return view


def evict_stats(h) -> dict:
    st = EvictStats()
    check(load().evict_stats(h, ctypes.byref(st)))
    return {f: getattr(st, f) for f, _ in EvictStats._fields_}


def evict_set_state(h, k_ptr, v_ptr, pos_ptr, score_ptr, n, offset):
    check(load().evict_set_state(h, k_ptr, v_ptr, pos_ptr, score_ptr, n, offset))


def evict_reset(h):
    check(load().evict_reset(h))


def evict_set_stream(h, stream):
    check(load().evict_set_stream(h, stream))


def evict_sync(h):
    check(load().evict_sync(h))


def evict_destroy(h):
    load().evict_destroy(h)


def evict_qfilters_calibrate(q_ptr, dtype, n_q_heads, n_samples, head_dim, n_kv_heads, out_ptr, stream):
    check(load().evict_qfilters_calibrate(q_ptr, dtype, n_q_heads, n_samples, head_dim, n_kv_heads, out_ptr,
                                          stream))


def evict_set_profiling(h, enable: bool):
    check(load().evict_set_profiling(h, int(enable)))


def evict_kernel_times(h) -> dict:
    buf = (EvictKernelTime * 32)()
    n = _I()
    check(load().evict_kernel_times(h, buf, 32, ctypes.byref(n)))
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n.value)}


def evict_compaction_rows(h):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    check(load().evict_compaction_rows(h, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def evict_prefill_noalloc(cfg: EvictConfig, k_ptr, v_ptr, pos_ptr, n, k_out, v_out, pos_out, score_out):
    """One-shot block eviction into caller buffers with no device allocation."""
    check(load().evict_prefill_noalloc(ctypes.byref(cfg), k_ptr, v_ptr, pos_ptr, n, k_out, v_out, pos_out,
                                       score_out))


def evict_noalloc_status(stream=None):
    """Synchronise `stream` and raise EvictError(EVICT_EDEVICE) if a no-allocation call's kernel
    reported an error since the last status call (the error word is then cleared)."""
    check(load().evict_noalloc_status(stream))


def evict_curdkv_scores(h, attn_ptr, lev_ptr) -> int:
    n = _I()
    check(load().evict_curdkv_scores(h, attn_ptr, lev_ptr, ctypes.byref(n)))
    return n.value


def evict_qfilters_filters(h):
    """Filters in use as a numpy fp32 array [rows, 128] (rows = 0 before a fallback freeze)."""
    import numpy as np
    n = _I()
    check(load().evict_qfilters_filters(h, None, ctypes.byref(n)))
    out = np.zeros((n.value, HEAD_DIM), np.float32)
    if n.value:
        check(load().evict_qfilters_filters(h, out.ctypes.data, ctypes.byref(n)))
    return out


def evict_launch_count() -> int:
    return load().evict_launch_count()


# --------------------------------------------------------------------------
# torch convenience wrapper
# --------------------------------------------------------------------------
class _CudaArray:
    """Exposes a device pointer to torch.as_tensor via __cuda_array_interface__."""

    def __init__(self, ptr, shape, typestr, strides=None):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": strides}


def view_tensors(view: EvictView, batch: int, heads: int, dtype: str):
    """Zero-copy torch tensors over a view: k, v [B,H,n,D], pos, score [B,H,n]."""
    import torch
    cap, n = view.capacity, view.n_kept
    esz = 2 if dtype == "bf16" else 4
    tstr = "<i2" if dtype == "bf16" else "<f4"
    kv_strides = (heads * cap * HEAD_DIM * esz, cap * HEAD_DIM * esz, HEAD_DIM * esz, esz)
    row_strides = (heads * cap * 4, cap * 4, 4)
    shp = (batch, heads, n, HEAD_DIM)

    def wrap(ptr, shape, ts, strides):
        return torch.as_tensor(_CudaArray(ptr, shape, ts, strides), device="cuda")

    k = wrap(view.k, shp, tstr, kv_strides)
    v = wrap(view.v, shp, tstr, kv_strides)
    if dtype == "bf16":
        k, v = k.view(torch.bfloat16), v.view(torch.bfloat16)
    pos = wrap(view.pos, (batch, heads, n), "<i4", row_strides)
    score = wrap(view.score, (batch, heads, n), "<f4", row_strides)
    return k, v, pos, score


class EvictCache:
    """One layer's cache on the current CUDA device (torch tensors in, views out)."""

    def __init__(self, method: str, batch: int, n_kv_heads: int, budget: int, n_sink: int = 4, recent: int = 0,
                 max_block: int = 8192, max_kept: int = 0, keep_low: bool = True, sign: int = 1, filters=None,
                 rank_cap: int = 16, dtype: str = "bf16", stream=None, calib_tokens: int = 128,
                 per_token: bool = False):
        import torch
        self.method, self.batch, self.heads, self.dtype = method, batch, n_kv_heads, dtype
        self._fallback = method == "qfilters" and filters is None
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self._filters = None
        cfg = EvictConfig(method=METHODS[method], dtype=DTYPES[dtype], batch=batch, n_kv_heads=n_kv_heads,
                          head_dim=HEAD_DIM, budget=budget, n_sink=n_sink, recent=recent, max_block=max_block,
                          max_kept=max_kept, keep_low=int(keep_low), sign=sign, filters=None,
                          n_filter_heads=0, rank_cap=rank_cap, stream=stream, calib_tokens=calib_tokens,
                          per_token=int(per_token))
        if filters is not None:
            f = torch.as_tensor(filters, dtype=torch.float32).cuda().contiguous()
            if f.dim() != 2 or f.shape[1] != HEAD_DIM:
                raise ValueError("filters must be [n_heads, 128]")
            self._filters = f
            cfg.filters = f.data_ptr()
            cfg.n_filter_heads = f.shape[0]
        self.handle = evict_init(cfg)
        self._filters = None        # the library copied them

    def close(self):
        if self.handle:
            evict_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def update_and_fetch(self, k, v, pos=None):
        m = k.shape[2]
        for t in (k, v):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("k and v must be contiguous CUDA tensors [B, H, m, 128]")
        pos_ptr = pos.data_ptr() if pos is not None else None
        view = evict_update_and_fetch(self.handle, k.data_ptr(), v.data_ptr(), pos_ptr, m)
        return view_tensors(view, self.batch, self.heads, self.dtype)

    def view(self):
        return view_tensors(evict_get_view(self.handle), self.batch, self.heads, self.dtype)

    def set_state(self, k, v, pos, score=None, offset=None):
        n = k.shape[2]
        evict_set_state(self.handle, k.data_ptr(), v.data_ptr(), pos.data_ptr(),
                        score.data_ptr() if score is not None else None, n, n if offset is None else offset)

    def reset(self):
        evict_reset(self.handle)

    def sync(self):
        evict_sync(self.handle)

    def stats(self):
        return evict_stats(self.handle)

    def filters(self):
        """Q-Filters: the filters in use, numpy [H, 128] calibrated or [B, H, 128] once the
        key-SVD fallback has frozen (None before)."""
        f = evict_qfilters_filters(self.handle)
        if f.shape[0] == 0:
            return None
        return f if f.shape[0] == self.heads and not self._fallback else f.reshape(self.batch, self.heads, HEAD_DIM)
