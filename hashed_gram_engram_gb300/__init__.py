"""GB300-native (sm_103a) forward of the DeepSeek-V4.1 Engram layer.

The compute lives in the CUDA library ``libengram_gb300.so`` (C ABI in
``include/engram.h``); this package only marshals arguments to it.  There
is no CPU or PyTorch fallback: without the built library every call raises.

    from hashed_gram_engram_gb300 import Engram
    layer = Engram(dim=4096, hc_mult=4, max_ngram_size=3, n_heads=8, head_dim=64,
                   max_tokens=64, table=table, rows=rows, row_offset=offsets, wkv=wkv,
                   q_weight=q, k_weight=k)
    out = layer.forward(hidden, hash_ids, token_mask)
"""
from __future__ import annotations

import numpy as np

from . import _lib
from ._lib import (EngramError, engram_config, engram_create, engram_debug_intermediates,
                   engram_debug_keep_value, engram_debug_staged_mx, engram_debug_staged_rows,
                   engram_destroy, engram_device_error,
                   engram_forward, engram_forward_host, engram_forward_host_flush,
                   engram_forward_host_pipelined, ENGRAM_HOST_DEFER_OUTPUT,
                   engram_gate_noalloc,
                   engram_last_error, engram_layout,
                   engram_lookup, engram_profile_enable, engram_profile_read,
                   engram_weights, ENGRAM_WKV_BF16, ENGRAM_WKV_MXFP8,
                   ENGRAM_TABLE_DEVICE, ENGRAM_TABLE_HOST_PINNED, ENGRAM_TABLE_FORMAT_BF16,
                   ENGRAM_TABLE_FORMAT_E4M3, ENGRAM_DEVERR_BAD_HASH_ID, ENGRAM_DEVERR_TIMEOUT,
                   engram_prefetch_create, engram_prefetch_destroy, engram_prefetch_forward,
                   engram_prefetch_join, engram_prefetch_pending, engram_prefetch_start)

__all__ = [
    "Engram", "EngramPrefetch", "EngramError", "engram_config", "engram_weights", "engram_create",
    "engram_destroy", "engram_lookup", "engram_forward", "engram_forward_host",
    "engram_forward_host_pipelined", "engram_forward_host_flush", "ENGRAM_HOST_DEFER_OUTPUT",
    "engram_gate_noalloc", "engram_debug_staged_mx", "engram_debug_keep_value",
    "engram_last_error", "engram_device_error", "engram_layout", "engram_debug_intermediates",
    "engram_debug_staged_rows", "engram_profile_enable", "engram_profile_read",
    "ENGRAM_WKV_BF16", "ENGRAM_WKV_MXFP8", "ENGRAM_TABLE_DEVICE",
    "ENGRAM_TABLE_HOST_PINNED", "ENGRAM_TABLE_FORMAT_BF16", "ENGRAM_TABLE_FORMAT_E4M3",
    "ENGRAM_DEVERR_BAD_HASH_ID", "ENGRAM_DEVERR_TIMEOUT",
    "engram_prefetch_create", "engram_prefetch_destroy", "engram_prefetch_start",
    "engram_prefetch_forward", "engram_prefetch_join", "engram_prefetch_pending",
]


def library_path() -> str:
    return _lib.LIB_PATH


class Engram:
    """One Engram layer bound to borrowed weights (class Engram's forward).

    Tensors are torch tensors on the handle's device (the table may be a
    pinned host tensor with ``table_location=ENGRAM_TABLE_HOST_PINNED``).
    An fp8 table is its e4m3 codes (uint8 [rows, head_dim]) as ``table`` and
    its ue8m0 scales (uint8 [rows, head_dim / 32]) as ``table_scale``.
    The object keeps references to them so they outlive the handle.
    """

    def __init__(self, *, dim, hc_mult, max_ngram_size, n_heads, head_dim, max_tokens,
                 table, rows, row_offset, wkv, q_weight, k_weight, wkv_scale=None,
                 eps=1e-6, clamp=1e-6, wkv_format=None, table_location=None, device=None,
                 keep_value=False, table_scale=None):
        import torch
        self.dim, self.hc_mult, self.head_dim = int(dim), int(hc_mult), int(head_dim)
        self.n_hash_cols = (int(max_ngram_size) - 1) * int(n_heads)
        self.max_tokens = int(max_tokens)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        # each column's first row in the table, as the caller laid it out
        # (engram_layout gives the bucket sizes and offsets of EngramLayout)
        row_offset = np.ascontiguousarray(np.asarray(row_offset, dtype=np.int64))
        if wkv_format is None:
            wkv_format = ENGRAM_WKV_MXFP8 if wkv_scale is not None else ENGRAM_WKV_BF16
        if table_location is None:
            table_location = ENGRAM_TABLE_DEVICE if table.is_cuda else ENGRAM_TABLE_HOST_PINNED
        if device is None:
            device = wkv.device.index if wkv.device.index is not None else torch.cuda.current_device()
        cfg = engram_config(dim=self.dim, hc_mult=self.hc_mult,
                            max_ngram_size=int(max_ngram_size), n_heads=int(n_heads),
                            head_dim=self.head_dim, eps=float(eps), clamp=float(clamp),
                            max_tokens=self.max_tokens, wkv_format=int(wkv_format),
                            table_location=int(table_location), device=int(device),
                            table_format=ENGRAM_TABLE_FORMAT_BF16 if table_scale is None
                            else ENGRAM_TABLE_FORMAT_E4M3)
        # the table's element type must match its declared format: the
        # kernels index rows by the format's row bytes, so a mismatch would
        # read past the end of the table
        n_rows = int(row_offset[-1] + rows[-1]) if len(rows) else 0
        if table_scale is None:
            if table.dtype != torch.bfloat16:
                raise ValueError("a bf16 table is expected (an fp8 table needs table_scale)")
        elif table.dtype != torch.uint8 or table_scale.dtype != torch.uint8:
            raise ValueError("an fp8 table is uint8 e4m3 codes with uint8 ue8m0 table_scale")
        if table.dim() != 2 or table.shape[1] != self.head_dim or table.shape[0] < n_rows or \
                not table.is_contiguous():
            raise ValueError(f"table must be contiguous [>= {n_rows}, {self.head_dim}]")
        if table_scale is not None and (table_scale.dim() != 2 or
                                        table_scale.shape[0] < n_rows or
                                        table_scale.shape[1] != self.head_dim // 32 or
                                        not table_scale.is_contiguous()):
            raise ValueError(f"table_scale must be contiguous [>= {n_rows}, {self.head_dim // 32}]")
        w = engram_weights(table=table.data_ptr(), row_offset=row_offset.ctypes.data,
                           rows=rows.ctypes.data, wkv=wkv.data_ptr(),
                           wkv_scale=None if wkv_scale is None else wkv_scale.data_ptr(),
                           q_weight=q_weight.data_ptr(), k_weight=k_weight.data_ptr(),
                           table_scale=None if table_scale is None else table_scale.data_ptr())
        self._keep = (table, table_scale, wkv, wkv_scale, q_weight, k_weight, rows, row_offset)
        self.device = int(device)
        self.handle = engram_create(cfg, w)
        if keep_value:  # validation: let intermediates() return the fused path's value
            engram_debug_keep_value(self.handle, 1)

    def close(self):
        if getattr(self, "handle", None):
            engram_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def lookup(self, hash_ids, background=False, stream=None):
        """Engram.prepare_embeddings: gather the rows of hash_ids [T, C]."""
        T = hash_ids.shape[0]
        engram_lookup(self.handle, hash_ids, hash_ids.stride(0) if T else self.n_hash_cols, T,
                      int(bool(background)), stream)

    def forward(self, hidden, hash_ids=None, token_mask=None, out=None, stream=None):
        """Engram.forward: returns hidden + gate * value (a new tensor unless out is given).

        hash_ids=None consumes the rows of the last lookup()."""
        import torch
        T = hidden.shape[0]
        if out is None:
            out = torch.empty_like(hidden)
        if stream is None:
            stream = torch.cuda.current_stream(hidden.device)
        ids_stride = hash_ids.stride(0) if hash_ids is not None and T else self.n_hash_cols
        mask = None
        if token_mask is not None:
            mask = token_mask if token_mask.dtype == torch.uint8 else token_mask.to(torch.uint8)
        engram_forward(self.handle, hidden, hidden.stride(), hash_ids, ids_stride, mask, out,
                       out.stride(), T, stream)
        return out

    __call__ = forward

    def forward_host(self, hidden_host, hash_ids_host, token_mask_host, out_host, stream=None):
        T = hidden_host.shape[0]
        engram_forward_host(self.handle, hidden_host, hash_ids_host, token_mask_host, out_host,
                            T, stream)

    def forward_host_pipelined(self, hidden_host, hash_ids_host, token_mask_host, out_host,
                               stream=None, defer_output=False):
        """forward_host whose input copies overlap the previous call (the host
        inputs must be ready when the call is made); with defer_output the
        output copy also overlaps the next call, and out_host is complete
        after the next call (or flush_host()) on the stream; see
        engram_forward_host_pipelined in include/engram.h."""
        T = hidden_host.shape[0]
        engram_forward_host_pipelined(self.handle, hidden_host, hash_ids_host, token_mask_host,
                                      out_host, T,
                                      ENGRAM_HOST_DEFER_OUTPUT if defer_output else 0, stream)

    def flush_host(self, stream=None):
        """The stream waits for the last pipelined call's output copy."""
        engram_forward_host_flush(self.handle, stream)

    def device_error(self, clear=True) -> int:
        return engram_device_error(self.handle, int(clear))

    def intermediates(self, T, stream=None):
        """fp32 gate [T, H] and value [T, D] of the last forward (validation hook)."""
        import torch
        dev = torch.device("cuda", self.device)
        gate = torch.empty((T, self.hc_mult), dtype=torch.float32, device=dev)
        value = torch.empty((T, self.dim), dtype=torch.float32, device=dev)
        engram_debug_intermediates(self.handle, gate, value, T, stream)
        return gate, value

    def staged_rows(self, T, stream=None):
        import torch
        rows = torch.empty((T, self.n_hash_cols * self.head_dim), dtype=torch.bfloat16,
                           device=torch.device("cuda", self.device))
        engram_debug_staged_rows(self.handle, rows, T, stream)
        return rows

    def wkv(self, hash_ids=None, stream=None, kv=None):
        """bf16 kv [T, N] (keys of copies 0..H-1, then the value) of hash_ids,
        or of the last lookup's rows; decode-sized T only."""
        import torch
        from ._lib import engram_wkv
        T = hash_ids.shape[0] if hash_ids is not None else None
        if T is None:
            raise ValueError("pass hash_ids, or kv sized for the staged T")
        N = (self.hc_mult + 1) * self.dim
        if kv is None:
            kv = torch.empty((T, N), dtype=torch.bfloat16,
                             device=torch.device("cuda", self.device))
        engram_wkv(self.handle, hash_ids, hash_ids.stride(0) if T else self.n_hash_cols, kv,
                   kv.stride(0), T, stream)
        return kv

    def staged_mx(self, T, stream=None):
        """e4m3 codes [T, K] and E8M0 scales [T, K/32] of the staged rows (MXFP8)."""
        import torch
        dev = torch.device("cuda", self.device)
        K = self.n_hash_cols * self.head_dim
        codes = torch.empty((T, K), dtype=torch.uint8, device=dev)
        scales = torch.empty((T, K // 32), dtype=torch.uint8, device=dev)
        engram_debug_staged_mx(self.handle, codes, scales, T, stream)
        return codes, scales


class EngramPrefetch:
    """Lookups of several layers run ahead on a side stream (class
    EngramPrefetch's start / forward / join on the prefetch page, with
    Engram.prepare_embeddings).  start() stages every layer's rows as soon
    as the step's hash ids exist; forward(i, ...) waits only for layer i's
    rows.  The layers must outlive this object; while it lives, only it
    looks up rows for them."""

    def __init__(self, layers, wkv=False):
        """wkv=True also runs each layer's projection on the side stream
        (where its fused decode launch serves T); forward then runs only the
        gate and residual."""
        self.layers = list(layers)
        self.handle = engram_prefetch_create([L.handle for L in self.layers],
                                             _lib.ENGRAM_PREFETCH_WKV if wkv else 0)
        self.T = None

    def close(self):
        if getattr(self, "handle", None):
            engram_prefetch_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream(self, stream):
        import torch
        if stream is not None:
            return stream
        return torch.cuda.current_stream(torch.device("cuda", self.layers[0].device))

    def start(self, hash_ids, background=True, stream=None):
        """hash_ids: one int32 [T, C] device tensor per layer (same T)."""
        assert len(hash_ids) == len(self.layers)
        T = int(hash_ids[0].shape[0])
        assert all(int(x.shape[0]) == T for x in hash_ids)
        strides = [x.stride(0) if T else L.n_hash_cols for x, L in zip(hash_ids, self.layers)]
        engram_prefetch_start(self.handle, hash_ids, strides, T, int(bool(background)),
                              self._stream(stream))
        self.T = T

    def forward(self, i, hidden, hash_ids=None, token_mask=None, out=None, stream=None):
        """Layer i's forward; hash_ids is needed only when nothing was staged
        ahead for it."""
        import torch
        T = hidden.shape[0]
        if out is None:
            out = torch.empty_like(hidden)
        ids_stride = hash_ids.stride(0) if hash_ids is not None and T else \
            self.layers[i].n_hash_cols
        mask = None
        if token_mask is not None:
            mask = token_mask if token_mask.dtype == torch.uint8 else token_mask.to(torch.uint8)
        engram_prefetch_forward(self.handle, i, hidden, hidden.stride(), hash_ids, ids_stride,
                                mask, out, out.stride(), T, self._stream(stream))
        return out

    def join(self, stream=None):
        engram_prefetch_join(self.handle, self._stream(stream))

    def pending(self, i) -> bool:
        return engram_prefetch_pending(self.handle, i)
