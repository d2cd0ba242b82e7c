"""ctypes binding of ``libengram_gb300.so`` (declared in ``include/engram.h``).

Argument marshalling only: every step of the forward runs in the CUDA
library.  Functions keep the C names.  Pointer arguments accept an int
address, ``None`` (NULL), or any object with ``data_ptr()`` (a torch tensor).
Streams accept an int handle, ``None`` (0), or an object with
``cuda_stream`` (a torch.cuda.Stream).  A non-zero return raises
``EngramError`` carrying the code.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libengram_gb300.so")

ENGRAM_OK = 0
ENGRAM_ERR_INVALID_ARG = -1
ENGRAM_ERR_UNSUPPORTED = -2
ENGRAM_ERR_T_EXCEEDS_MAX = -3
ENGRAM_ERR_OOM = -4
ENGRAM_ERR_NO_UVA = -5
ENGRAM_ERR_DEVICE = -6
ENGRAM_ERR_CUDA = -7
ENGRAM_ERR_SCRATCH_LIMIT = -8
ERROR_NAMES = {
    -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "T_EXCEEDS_MAX", -4: "OOM", -5: "NO_UVA",
    -6: "DEVICE", -7: "CUDA", -8: "SCRATCH_LIMIT",
}
ENGRAM_NOALLOC_MAX_PARTIALS = 131072
ENGRAM_DEVERR_BAD_HASH_ID = 1
ENGRAM_DEVERR_TIMEOUT = 2
ENGRAM_WKV_BF16 = 0
ENGRAM_WKV_MXFP8 = 1
ENGRAM_TABLE_DEVICE = 0
ENGRAM_TABLE_HOST_PINNED = 1
ENGRAM_TABLE_FORMAT_BF16 = 0
ENGRAM_TABLE_FORMAT_E4M3 = 1
ENGRAM_FUSED_PLAN_FIELDS = 16
ENGRAM_HOST_DEFER_OUTPUT = 1

# Every symbol include/engram.h declares.
EXPORTED = (
    "engram_create", "engram_destroy", "engram_lookup", "engram_forward",
    "engram_forward_host", "engram_forward_host_pipelined", "engram_forward_host_flush",
    "engram_last_error",
    "engram_device_error", "engram_layout",
    "engram_debug_intermediates", "engram_debug_staged_rows", "engram_profile_enable",
    "engram_profile_read", "engram_gate_noalloc", "engram_debug_staged_mx",
    "engram_debug_fused_plan",
    "engram_debug_keep_value",
    "engram_prefetch_create", "engram_prefetch_destroy", "engram_prefetch_start",
    "engram_prefetch_forward", "engram_prefetch_join", "engram_prefetch_pending",
    "engram_debug_barrier_skew",
    "engram_wkv",
)


class EngramError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: ENGRAM_ERR_{ERROR_NAMES.get(code, code)} ({code})")


class engram_config(ctypes.Structure):
    _fields_ = [
        ("dim", ctypes.c_int64), ("hc_mult", ctypes.c_int64),
        ("max_ngram_size", ctypes.c_int64), ("n_heads", ctypes.c_int64),
        ("head_dim", ctypes.c_int64), ("eps", ctypes.c_double), ("clamp", ctypes.c_double),
        ("max_tokens", ctypes.c_int64), ("wkv_format", ctypes.c_int32),
        ("table_location", ctypes.c_int32), ("device", ctypes.c_int32),
        ("table_format", ctypes.c_int32),
    ]


class engram_weights(ctypes.Structure):
    _fields_ = [
        ("table", ctypes.c_void_p), ("row_offset", ctypes.c_void_p), ("rows", ctypes.c_void_p),
        ("wkv", ctypes.c_void_p), ("wkv_scale", ctypes.c_void_p),
        ("q_weight", ctypes.c_void_p), ("k_weight", ctypes.c_void_p),
        ("table_scale", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        sig = {
            "engram_create": [vp, vp, vp],
            "engram_destroy": [vp],
            "engram_lookup": [vp, vp, i64, i64, ctypes.c_int, vp],
            "engram_forward": [vp, vp, vp, vp, i64, vp, vp, vp, i64, vp],
            "engram_forward_host": [vp, vp, vp, vp, vp, i64, vp],
            "engram_forward_host_pipelined": [vp, vp, vp, vp, vp, i64, ctypes.c_uint32, vp],
            "engram_forward_host_flush": [vp, vp],
            "engram_last_error": [vp, ctypes.c_int],
            "engram_device_error": [vp, vp, ctypes.c_int],
            "engram_layout": [i64, i32, i32, i32, vp, vp],
            "engram_debug_intermediates": [vp, vp, vp, i64, vp],
            "engram_debug_staged_rows": [vp, vp, i64, vp],
            "engram_debug_staged_mx": [vp, vp, vp, i64, vp],
            "engram_debug_fused_plan": [vp, i64, i32, vp, i32],
            "engram_debug_keep_value": [vp, ctypes.c_int],
            "engram_profile_enable": [vp, ctypes.c_int],
            "engram_profile_read": [vp, vp],
            "engram_gate_noalloc": [vp, vp, vp, i64, vp, vp, vp, vp, vp, i64, i64, i64,
                                    ctypes.c_double, ctypes.c_double, vp],
            "engram_debug_barrier_skew": [vp, i64],
            "engram_prefetch_create": [vp, i32, i32, vp],
            "engram_wkv": [vp, vp, i64, vp, i64, i64, vp],
            "engram_prefetch_destroy": [vp],
            "engram_prefetch_start": [vp, vp, vp, i64, ctypes.c_int, vp],
            "engram_prefetch_forward": [vp, i32, vp, vp, vp, i64, vp, vp, vp, i64, vp],
            "engram_prefetch_join": [vp, vp],
            "engram_prefetch_pending": [vp, i32],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        _lib = L
        return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr() if x.numel() > 0 else None
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc, what):
    if rc != ENGRAM_OK:
        raise EngramError(rc, what)
    return rc


def _i64x3(v):
    return None if v is None else (ctypes.c_int64 * 3)(*[int(x) for x in v])


def engram_create(cfg: engram_config, weights: engram_weights) -> int:
    h = ctypes.c_void_p()
    _check(load().engram_create(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(h)),
           "engram_create")
    return h.value


def engram_destroy(h: int) -> None:
    _check(load().engram_destroy(h), "engram_destroy")


def engram_lookup(h, hash_ids, ids_row_stride, T, background=0, stream=None):
    return _check(load().engram_lookup(h, _ptr(hash_ids), int(ids_row_stride), int(T),
                                       int(background), _stream(stream)), "engram_lookup")


def engram_forward(h, hidden, hidden_strides, hash_ids, ids_row_stride, token_mask, out,
                   out_strides, T, stream=None):
    return _check(load().engram_forward(
        h, _ptr(hidden), _i64x3(hidden_strides), _ptr(hash_ids), int(ids_row_stride),
        _ptr(token_mask), _ptr(out), _i64x3(out_strides), int(T), _stream(stream)),
        "engram_forward")


def engram_forward_host(h, hidden_host, hash_ids_host, token_mask_host, out_host, T,
                        stream=None):
    return _check(load().engram_forward_host(
        h, _ptr(hidden_host), _ptr(hash_ids_host), _ptr(token_mask_host), _ptr(out_host),
        int(T), _stream(stream)), "engram_forward_host")


def engram_forward_host_pipelined(h, hidden_host, hash_ids_host, token_mask_host, out_host, T,
                                  flags=0, stream=None):
    return _check(load().engram_forward_host_pipelined(
        h, _ptr(hidden_host), _ptr(hash_ids_host), _ptr(token_mask_host), _ptr(out_host),
        int(T), int(flags), _stream(stream)), "engram_forward_host_pipelined")


def engram_forward_host_flush(h, stream=None):
    return _check(load().engram_forward_host_flush(h, _stream(stream)),
                  "engram_forward_host_flush")


def engram_last_error(h, sync=0) -> int:
    return load().engram_last_error(h, int(sync))


def engram_device_error(h, clear=1) -> int:
    bits = ctypes.c_uint32()
    _check(load().engram_device_error(h, ctypes.byref(bits), int(clear)), "engram_device_error")
    return bits.value


def engram_layout(vocab_size, max_ngram_size, n_heads, n_layers=1):
    cols = (max_ngram_size - 1) * n_heads
    primes = (ctypes.c_int64 * (cols * n_layers))()
    offsets = (ctypes.c_int64 * (cols * n_layers))()
    _check(load().engram_layout(int(vocab_size), int(max_ngram_size), int(n_heads),
                                int(n_layers), primes, offsets), "engram_layout")
    return ([list(primes[l * cols:(l + 1) * cols]) for l in range(n_layers)],
            [list(offsets[l * cols:(l + 1) * cols]) for l in range(n_layers)])


FUSED_PLAN_KEYS = ("used", "grid", "max_width", "mtiles", "k_blocks", "w_stages", "x_stages",
                   "w_stage_bytes", "x_stage_bytes", "x_off", "x_ring", "qk_off", "bar_off",
                   "smem_bytes", "dual", "Tn")


def engram_debug_fused_plan(cfg, T, num_sms):
    """The fused decode kernel's plan for cfg, T and num_sms (host only)."""
    out = (ctypes.c_int64 * ENGRAM_FUSED_PLAN_FIELDS)()
    _check(load().engram_debug_fused_plan(ctypes.byref(cfg), int(T), int(num_sms), out,
                                          ENGRAM_FUSED_PLAN_FIELDS), "engram_debug_fused_plan")
    return dict(zip(FUSED_PLAN_KEYS, list(out)))


def engram_debug_intermediates(h, gate, value, T, stream=None):
    return _check(load().engram_debug_intermediates(h, _ptr(gate), _ptr(value), int(T),
                                                    _stream(stream)),
                  "engram_debug_intermediates")


def engram_debug_staged_rows(h, rows, T, stream=None):
    return _check(load().engram_debug_staged_rows(h, _ptr(rows), int(T), _stream(stream)),
                  "engram_debug_staged_rows")


def engram_debug_staged_mx(h, codes, scales, T, stream=None):
    return _check(load().engram_debug_staged_mx(h, _ptr(codes), _ptr(scales), int(T),
                                                _stream(stream)), "engram_debug_staged_mx")


def engram_debug_keep_value(h, enable=1):
    return _check(load().engram_debug_keep_value(h, int(enable)), "engram_debug_keep_value")


def engram_profile_enable(h, enable=1):
    return _check(load().engram_profile_enable(h, int(enable)), "engram_profile_enable")


def engram_profile_read(h):
    ms = (ctypes.c_float * 3)()
    _check(load().engram_profile_read(h, ms), "engram_profile_read")
    return list(ms)


def engram_gate_noalloc(hidden, hidden_strides, kv, kv_row_stride, q_weight, k_weight,
                        token_mask, out, out_strides, T, H, D, eps=1e-6, clamp=1e-6,
                        stream=None):
    """Gate + masked residual over a caller-computed kv, no handle, no allocation."""
    return _check(load().engram_gate_noalloc(
        _ptr(hidden), _i64x3(hidden_strides), _ptr(kv), int(kv_row_stride), _ptr(q_weight),
        _ptr(k_weight), _ptr(token_mask), _ptr(out), _i64x3(out_strides), int(T), int(H),
        int(D), float(eps), float(clamp), _stream(stream)), "engram_gate_noalloc")


ENGRAM_PREFETCH_WKV = 1


def engram_prefetch_create(handles, flags=0) -> int:
    arr = (ctypes.c_void_p * len(handles))(*handles)
    p = ctypes.c_void_p()
    _check(load().engram_prefetch_create(arr, len(handles), int(flags), ctypes.byref(p)),
           "engram_prefetch_create")
    return p.value


def engram_wkv(h, hash_ids, ids_row_stride, kv, kv_row_stride, T, stream=None):
    return _check(load().engram_wkv(h, _ptr(hash_ids), int(ids_row_stride), _ptr(kv),
                                    int(kv_row_stride), int(T), _stream(stream)), "engram_wkv")


def engram_prefetch_destroy(p) -> None:
    _check(load().engram_prefetch_destroy(p), "engram_prefetch_destroy")


def engram_prefetch_start(p, hash_ids, ids_row_strides, T, background=1, stream=None):
    n = len(hash_ids)
    ids = (ctypes.c_void_p * n)(*[_ptr(x) for x in hash_ids])
    st = (ctypes.c_int64 * n)(*[int(x) for x in ids_row_strides])
    return _check(load().engram_prefetch_start(p, ids, st, int(T), int(background),
                                               _stream(stream)), "engram_prefetch_start")


def engram_prefetch_forward(p, layer, hidden, hidden_strides, hash_ids, ids_row_stride,
                            token_mask, out, out_strides, T, stream=None):
    return _check(load().engram_prefetch_forward(
        p, int(layer), _ptr(hidden), _i64x3(hidden_strides), _ptr(hash_ids),
        int(ids_row_stride), _ptr(token_mask), _ptr(out), _i64x3(out_strides), int(T),
        _stream(stream)), "engram_prefetch_forward")


def engram_prefetch_join(p, stream=None):
    return _check(load().engram_prefetch_join(p, _stream(stream)), "engram_prefetch_join")


def engram_prefetch_pending(p, layer) -> bool:
    rc = load().engram_prefetch_pending(p, int(layer))
    if rc < 0:
        _check(rc, "engram_prefetch_pending")
    return rc == 1


def engram_debug_barrier_skew(h, delta):
    return _check(load().engram_debug_barrier_skew(h, int(delta)), "engram_debug_barrier_skew")
