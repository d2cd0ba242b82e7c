"""numpy wrappers over the C oracle (``engram_oracle.c``).  Test infrastructure only.

Each wrapper states the page passage its C function follows; the C file
carries the full citations.  Arrays are passed as raw numpy buffers: bf16
data travels as ``uint16`` bit patterns, e4m3 and E8M0 as ``uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "build_oracle", "lib", "bf16_to_f64", "e4m3_to_f64", "e8m0_to_f64",
    "f64_to_e4m3", "f64_to_bf16", "layout", "gather", "gather_e4m3", "wkv_bf16", "wkv_mxfp8",
    "mx_quantize", "wkv_mxfp8_qact", "gate", "forward",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "engram_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, portable flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build_oracle())
            vp, i64, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = f64
            L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_f64.restype = f64
            L.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
            L.oracle_e8m0_to_f64.restype = f64
            L.oracle_f64_to_e4m3_satfinite.argtypes = [f64]
            L.oracle_f64_to_e4m3_satfinite.restype = ctypes.c_uint8
            L.oracle_f64_to_bf16.argtypes = [f64]
            L.oracle_f64_to_bf16.restype = ctypes.c_uint16
            L.oracle_layout.argtypes = [i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
            L.oracle_layout.restype = ctypes.c_int
            L.oracle_gather.argtypes = [vp, vp, vp, i64, i64, vp, i64, i64, vp, vp]
            L.oracle_gather.restype = None
            L.oracle_gather_e4m3.argtypes = [vp, vp, vp, vp, i64, i64, vp, i64, i64, vp, vp]
            L.oracle_gather_e4m3.restype = None
            L.oracle_wkv_bf16.argtypes = [vp, i64, i64, vp, i64, vp]
            L.oracle_wkv_bf16.restype = None
            L.oracle_wkv_mxfp8.argtypes = [vp, i64, i64, vp, vp, i64, vp]
            L.oracle_wkv_mxfp8.restype = None
            L.oracle_mx_quantize.argtypes = [vp, i64, i64, vp, vp]
            L.oracle_mx_quantize.restype = None
            L.oracle_wkv_mxfp8_qact.argtypes = [vp, vp, i64, i64, vp, vp, i64, vp]
            L.oracle_wkv_mxfp8_qact.restype = None
            L.oracle_gate.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, f64, f64,
                                      vp, vp, vp, vp]
            L.oracle_gate.restype = None
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


# -- number formats ---------------------------------------------------------

def bf16_to_f64(bits):
    L = lib()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([L.oracle_bf16_to_f64(int(x)) for x in b.ravel()]).reshape(b.shape)


def e4m3_to_f64(codes):
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.oracle_e4m3_to_f64(int(x)) for x in c.ravel()]).reshape(c.shape)


def e8m0_to_f64(b):
    L = lib()
    b = np.asarray(b, dtype=np.uint8)
    return np.array([L.oracle_e8m0_to_f64(int(x)) for x in b.ravel()]).reshape(b.shape)


def f64_to_e4m3(x):
    L = lib()
    x = np.asarray(x, dtype=np.float64)
    return np.array([L.oracle_f64_to_e4m3_satfinite(float(v)) for v in x.ravel()],
                    dtype=np.uint8).reshape(x.shape)


def f64_to_bf16(x):
    L = lib()
    x = np.asarray(x, dtype=np.float64)
    return np.array([L.oracle_f64_to_bf16(float(v)) for v in x.ravel()],
                    dtype=np.uint16).reshape(x.shape)


# -- EngramLayout -------------------------------------------------------------

def layout(vocab_size: int, max_ngram_size: int, n_heads: int, n_layers: int = 1):
    """Prime bucket sizes and offsets per layer (class EngramLayout)."""
    cols = (max_ngram_size - 1) * n_heads
    primes = np.zeros((n_layers, cols), np.int64)
    offsets = np.zeros((n_layers, cols), np.int64)
    rc = lib().oracle_layout(vocab_size, max_ngram_size, n_heads, n_layers,
                             _p(primes), _p(offsets))
    if rc != 0:
        raise ValueError("bad layout arguments")
    return primes, offsets


# -- forward steps ---------------------------------------------------------------

def gather(table_bits, row_offset, rows, ids, E):
    """rows[t, c, :] = table[row_offset[c] + ids[t, c]] (ParallelEngramEmbedding.lookup).

    Returns (rows uint16 [T, C, E], number of out-of-range ids)."""
    table_bits = _c(table_bits, np.uint16)
    row_offset = _c(np.asarray(row_offset, np.int64), np.int64)
    rows = _c(np.asarray(rows, np.int64), np.int64)
    ids = np.asarray(ids)
    assert ids.dtype == np.int32 and ids.ndim == 2 and ids.strides[1] == 4
    T, C = ids.shape
    stride = ids.strides[0] // 4 if T > 0 else C
    out = np.zeros((T, C, E), np.uint16)
    nbad = np.zeros(1, np.int64)
    base = ids if ids.flags.c_contiguous else ids
    lib().oracle_gather(_p(table_bits), _p(row_offset), _p(rows), C, E,
                        ctypes.c_void_p(base.ctypes.data), stride, T, _p(out), _p(nbad))
    return out, int(nbad[0])


def gather_e4m3(codes, scales, row_offset, rows, ids, E):
    """gather() from an fp8 table: e4m3 codes [total_rows, E] with one ue8m0
    scale byte per 32 elements [total_rows, E / 32], dequantized to bf16 bits
    (class ParallelEngramEmbedding).  Returns (rows uint16 [T, C, E], bad ids)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    assert E % 32 == 0 and codes.shape[-1] == E and scales.shape[-1] == E // 32
    row_offset = _c(np.asarray(row_offset, np.int64), np.int64)
    rows = _c(np.asarray(rows, np.int64), np.int64)
    ids = np.asarray(ids)
    assert ids.dtype == np.int32 and ids.ndim == 2 and ids.strides[1] == 4
    T, C = ids.shape
    stride = ids.strides[0] // 4 if T > 0 else C
    out = np.zeros((T, C, E), np.uint16)
    nbad = np.zeros(1, np.int64)
    lib().oracle_gather_e4m3(_p(codes), _p(scales), _p(row_offset), _p(rows), C, E,
                             ctypes.c_void_p(ids.ctypes.data), stride, T, _p(out), _p(nbad))
    return out, int(nbad[0])


def wkv_bf16(A_bits, W_bits):
    """kv = A . W^T in fp64 (Engram.forward's wkv on the flattened rows)."""
    A_bits = _c(A_bits, np.uint16)
    W_bits = _c(W_bits, np.uint16)
    T, K = A_bits.shape
    N = W_bits.shape[0]
    assert W_bits.shape[1] == K
    kv = np.zeros((T, N), np.float64)
    lib().oracle_wkv_bf16(_p(A_bits), T, K, _p(W_bits), N, _p(kv))
    return kv


def wkv_mxfp8(A_bits, Wq, Ws):
    """kv = A . dequant(W)^T with MXFP8 e4m3 weights and E8M0 32x32 scales."""
    A_bits = _c(A_bits, np.uint16)
    Wq = _c(Wq, np.uint8)
    Ws = _c(Ws, np.uint8)
    T, K = A_bits.shape
    N = Wq.shape[0]
    assert Wq.shape[1] == K and Ws.shape == (N // 32, K // 32)
    kv = np.zeros((T, N), np.float64)
    lib().oracle_wkv_mxfp8(_p(A_bits), T, K, _p(Wq), _p(Ws), N, _p(kv))
    return kv


def mx_quantize(A_bits):
    """MXFP8 activation quantisation: per 32 k, power-of-two scale, e4m3 RTNE."""
    A_bits = _c(A_bits, np.uint16)
    T, K = A_bits.shape
    codes = np.zeros((T, K), np.uint8)
    scales = np.zeros((T, K // 32), np.uint8)
    lib().oracle_mx_quantize(_p(A_bits), T, K, _p(codes), _p(scales))
    return codes, scales


def wkv_mxfp8_qact(Aq, As, Wq, Ws):
    Aq = _c(Aq, np.uint8)
    As = _c(As, np.uint8)
    Wq = _c(Wq, np.uint8)
    Ws = _c(Ws, np.uint8)
    T, K = Aq.shape
    N = Wq.shape[0]
    kv = np.zeros((T, N), np.float64)
    lib().oracle_wkv_mxfp8_qact(_p(Aq), _p(As), T, K, _p(Wq), _p(Ws), N, _p(kv))
    return kv


def gate(hidden_bits, kv, q_bits, k_bits, mask, eps=1e-6, clamp=1e-6):
    """Gate and masked residual (Engram.forward; the finish kernel at one rank).

    hidden_bits: uint16 [T, H, D] (any strides, unit dim stride not required).
    Returns dict(out_f64, out_bf16, gate, dot)."""
    hidden_bits = np.asarray(hidden_bits)
    assert hidden_bits.dtype == np.uint16 and hidden_bits.ndim == 3
    T, H, D = hidden_bits.shape
    hs = np.array([s // 2 for s in hidden_bits.strides], np.int64)
    kv = _c(kv, np.float64)
    assert kv.shape == (T, (H + 1) * D)
    q_bits = _c(q_bits, np.uint16)
    k_bits = _c(k_bits, np.uint16)
    m = None if mask is None else _c(np.asarray(mask).astype(np.uint8), np.uint8)
    out_f64 = np.zeros((T, H, D), np.float64)
    out_bf16 = np.zeros((T, H, D), np.uint16)
    g = np.zeros((T, H), np.float64)
    dot = np.zeros((T, H), np.float64)
    lib().oracle_gate(ctypes.c_void_p(hidden_bits.ctypes.data), _p(hs), _p(kv),
                      _p(q_bits), _p(k_bits), _p(m), T, H, D, float(eps), float(clamp),
                      _p(out_f64), _p(out_bf16), _p(g), _p(dot))
    return dict(out_f64=out_f64, out_bf16=out_bf16, gate=g, dot=dot)


def forward(table_bits, row_offset, rows, ids, E, W, hidden_bits, q_bits, k_bits,
            mask=None, Ws=None, eps=1e-6, clamp=1e-6, quantize_act=False, table_scale=None):
    """The whole layer: gather -> wkv -> gate/residual.

    The table is bf16 bits, or (table_scale given) e4m3 codes with one ue8m0
    scale per 32 elements.  W is bf16 bits [N, K] (Ws None) or e4m3 codes
    with E8M0 scales Ws.  With quantize_act the MXFP8 path quantises the
    rows first.  Returns the gate() dict plus rows, kv and the bad-id count."""
    if table_scale is None:
        rws, nbad = gather(table_bits, row_offset, rows, ids, E)
    else:
        rws, nbad = gather_e4m3(table_bits, table_scale, row_offset, rows, ids, E)
    T, C, _ = rws.shape
    A = rws.reshape(T, C * E)
    if Ws is None:
        kv = wkv_bf16(A, W)
    elif quantize_act:
        Aq, As = mx_quantize(A)
        kv = wkv_mxfp8_qact(Aq, As, W, Ws)
    else:
        kv = wkv_mxfp8(A, W, Ws)
    res = gate(hidden_bits, kv, q_bits, k_bits, mask, eps, clamp)
    res.update(rows=rws, kv=kv, n_bad=nbad)
    return res
