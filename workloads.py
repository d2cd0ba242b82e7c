"""Seeded synthetic inputs for the Engram forward, shared by the tests, the
benchmark and the smoke check.

This module only draws random numbers and lays them out; it holds none of
the layer's arithmetic.  Shapes, value distributions and id skew follow the
workloads the Engram layer runs on (DeepSeek-V4.1 decode and prefill steps,
an MXFP8 wkv, and host-offloaded tables):

* table rows, wkv, q_weight, k_weight: bf16 N(0, 0.02)
* hidden: bf16 N(0, 1), [T, hc_mult, dim], contiguous
* MXFP8 wkv: e4m3 codes of N(0, 1) (torch's float8_e4m3fn cast) with E8M0
  scale bytes uniform in {119..127} (block exponents -8..0)
* fp8 tables (e4m3 rows, one ue8m0 scale per 32 elements, the storage of
  class ParallelEngramEmbedding): codes of N(0, 1) the same way, scale bytes
  uniform in {113..121} (exponents -14..-6, magnitudes near the bf16 tables')
* hash ids: per column local ids, uniform over [0, rows[c]), or Zipf(1.1)
  ranks scattered over the rows by a per-column bijection r -> (a r + b) mod p
* token_mask: Bernoulli(p) bytes, or None

Table sizes: the bucket sizes of class EngramLayout (next primes above
engram_vocab_size - 1, none reused): 2^19 for the decode-shaped configs,
2^23 for the offloaded one.  The tiny config uses a fixed list of eight
primes between 1009 and 1103.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np
import torch

# EngramLayout bucket sizes (class EngramLayout.__init__): 2 n-gram orders x
# 8 heads from engram_vocab_size = 2^19 and 2^23.
PRIMES_2POW19 = (524309, 524341, 524347, 524351, 524353, 524369, 524387, 524389,
                 524411, 524413, 524429, 524453, 524497, 524507, 524509, 524519)
PRIMES_2POW23 = (8388617, 8388619, 8388623, 8388637, 8388673, 8388683, 8388691,
                 8388697, 8388733, 8388739, 8388761, 8388763, 8388791, 8388811,
                 8388833, 8388841)
TINY_ROWS = (1009, 1019, 1033, 1049, 1061, 1069, 1093, 1103)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    dim: int
    hc_mult: int
    max_ngram_size: int
    n_heads: int
    head_dim: int
    rows: tuple
    wkv_format: str = "bf16"        # "bf16" | "mxfp8"
    ids: str = "uniform"            # "uniform" | "zipf"
    mask_p: float | None = None     # Bernoulli(p) token mask, None = no mask
    table_location: str = "device"  # "device" | "host"
    table_format: str = "bf16"      # "bf16" | "e4m3" (with ue8m0 scales per 32)
    tol: float = 3e-2               # max abs error on the output
    seed: int = 1234
    eps: float = 1e-6
    clamp: float = 1e-6

    @property
    def n_hash_cols(self) -> int:
        return (self.max_ngram_size - 1) * self.n_heads

    @property
    def K(self) -> int:
        return self.n_hash_cols * self.head_dim

    @property
    def N(self) -> int:
        return self.dim * (self.hc_mult + 1)

    @property
    def total_rows(self) -> int:
        return int(sum(self.rows))

    def with_T(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T)


TINY = Workload("tiny", T=16, dim=256, hc_mult=2, max_ngram_size=3, n_heads=4,
                head_dim=32, rows=TINY_ROWS, mask_p=0.75, tol=2e-2, seed=1234)
DECODE = Workload("decode", T=64, dim=4096, hc_mult=4, max_ngram_size=3, n_heads=8,
                  head_dim=64, rows=PRIMES_2POW19, tol=3e-2, seed=1235)
PREFILL = Workload("prefill", T=8192, dim=4096, hc_mult=4, max_ngram_size=3,
                   n_heads=8, head_dim=64, rows=PRIMES_2POW19, ids="zipf",
                   mask_p=0.9, tol=3e-2, seed=1236)
MXFP8_DECODE = Workload("mxfp8_decode", T=64, dim=7168, hc_mult=4, max_ngram_size=3,
                        n_heads=8, head_dim=64, rows=PRIMES_2POW19, wkv_format="mxfp8",
                        tol=5e-2, seed=1237)
MXFP8_PREFILL = dataclasses.replace(MXFP8_DECODE, name="mxfp8_prefill", T=4096,
                                    seed=1238)
OFFLOAD = Workload("offload", T=256, dim=4096, hc_mult=4, max_ngram_size=3, n_heads=8,
                   head_dim=64, rows=PRIMES_2POW23, table_location="host", tol=3e-2,
                   seed=1239)

# parity case only (not a benchmark configuration): the tiny shapes with MXFP8 wkv
TINY_MXFP8 = dataclasses.replace(TINY, name="tiny_mxfp8", wkv_format="mxfp8", tol=5e-2,
                                 seed=1240)
# fp8 (e4m3 + ue8m0 per 32) tables, the storage the pages' ParallelEngramEmbedding
# keeps: the decode and offload shapes, and a tiny parity case
DECODE_E4M3 = dataclasses.replace(DECODE, name="decode_e4m3_table", table_format="e4m3",
                                  seed=1241)
OFFLOAD_E4M3 = dataclasses.replace(OFFLOAD, name="offload_e4m3_table", table_format="e4m3",
                                   seed=1242)
TINY_E4M3 = dataclasses.replace(TINY, name="tiny_e4m3_table", table_format="e4m3", seed=1243)
ALL = {w.name: w for w in (TINY, DECODE, PREFILL, MXFP8_DECODE, MXFP8_PREFILL, OFFLOAD,
                           DECODE_E4M3, OFFLOAD_E4M3)}


def shard_tokens(T: int, rank: int, world: int) -> tuple[int, int]:
    """Token range [lo, hi) of one rank when T tokens are split evenly (the
    forward has no cross-token dependence, so ranks need no exchange)."""
    return T * rank // world, T * (rank + 1) // world


def row_offsets(rows) -> np.ndarray:
    """Start row of every column's bucket in the concatenated table."""
    r = np.asarray(rows, np.int64)
    return np.concatenate([[0], np.cumsum(r)[:-1]]).astype(np.int64)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, std, g, device):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            * std).to(torch.bfloat16)


def _e4m3_codes(shape, g, device):
    return torch.randn(shape, generator=g, device=device).to(torch.float8_e4m3fn).view(
        torch.uint8)


def make_table(wl: Workload, device="cpu", chunk_rows=1 << 22):
    """bf16 [total_rows, head_dim] N(0, 0.02), or for an e4m3 table its codes
    (uint8, same shape).  For table_location "host" the rows are drawn on
    ``device`` in chunks and stored in pinned host memory."""
    g = _gen(device, wl.seed * 7 + 1)
    n, E = wl.total_rows, wl.head_dim
    fp8 = wl.table_format == "e4m3"
    dt = torch.uint8 if fp8 else torch.bfloat16
    draw = (lambda m: _e4m3_codes((m, E), g, device)) if fp8 else (
        lambda m: _normal_bf16((m, E), 0.02, g, device))
    if wl.table_location == "host":
        out = torch.empty((n, E), dtype=dt, pin_memory=True)
        for s in range(0, n, chunk_rows):
            e = min(n, s + chunk_rows)
            out[s:e].copy_(draw(e - s))
        return out
    out = torch.empty((n, E), dtype=dt, device=device)
    for s in range(0, n, chunk_rows):
        e = min(n, s + chunk_rows)
        out[s:e] = draw(e - s)
    return out


def make_table_scale(wl: Workload, device="cpu"):
    """ue8m0 scale bytes [total_rows, head_dim / 32] of an e4m3 table, uniform
    in {113..121} (in pinned host memory for table_location "host"); None for
    a bf16 table."""
    if wl.table_format != "e4m3":
        return None
    g = _gen(device, wl.seed * 7 + 5)
    sc = torch.randint(113, 122, (wl.total_rows, wl.head_dim // 32), generator=g,
                       device=device, dtype=torch.int32).to(torch.uint8)
    if wl.table_location == "host":
        out = torch.empty(sc.shape, dtype=torch.uint8, pin_memory=True)
        out.copy_(sc)
        return out
    return sc


def make_weights(wl: Workload, device="cpu"):
    """wkv (bf16 [N, K], or e4m3 codes [N, K] + E8M0 [N/32, K/32]), q, k."""
    g = _gen(device, wl.seed * 7 + 2)
    N, K, H, D = wl.N, wl.K, wl.hc_mult, wl.dim
    if wl.wkv_format == "mxfp8":
        codes = torch.randn((N, K), generator=g, device=device).to(
            torch.float8_e4m3fn).view(torch.uint8)
        scales = torch.randint(119, 128, (N // 32, K // 32), generator=g,
                               device=device, dtype=torch.int32).to(torch.uint8)
        wkv, wkv_scale = codes, scales
    else:
        wkv, wkv_scale = _normal_bf16((N, K), 0.02, g, device), None
    q = _normal_bf16((H, D), 0.02, g, device)
    k = _normal_bf16((H, D), 0.02, g, device)
    return dict(wkv=wkv, wkv_scale=wkv_scale, q_weight=q, k_weight=k)


def _zipf_ids(rows, T, rng):
    cols = []
    for c, p in enumerate(rows):
        w = np.arange(1, p + 1, dtype=np.float64) ** -1.1
        cdf = np.cumsum(w)
        cdf /= cdf[-1]
        r = np.searchsorted(cdf, rng.random(T), side="right")
        r = np.minimum(r, p - 1)
        a = (2654435761 % p) or 1
        b = (7919 * (c + 1) + 13) % p
        cols.append((a * r + b) % p)
    return np.stack(cols, axis=1).astype(np.int32)


def make_step_inputs(wl: Workload, device="cpu", T: int | None = None, step: int = 0):
    """hidden [T, H, D] bf16, hash_ids int32 [T, C], token_mask uint8 [T] | None."""
    T = wl.T if T is None else T
    seed = wl.seed * 7 + 3 + 1000 * step
    g = _gen(device, seed)
    hidden = _normal_bf16((T, wl.hc_mult, wl.dim), 1.0, g, device)
    if wl.ids == "zipf":
        ids = torch.from_numpy(_zipf_ids(wl.rows, T, np.random.default_rng(seed))).to(device)
    else:
        hi = torch.tensor(wl.rows, dtype=torch.float64, device=device)
        u = torch.rand((T, wl.n_hash_cols), generator=g, device=device, dtype=torch.float64)
        ids = torch.minimum((u * hi).floor(), hi - 1).to(torch.int32)
    mask = None
    if wl.mask_p is not None:
        mask = (torch.rand((T,), generator=g, device=device) < wl.mask_p).to(torch.uint8)
    return dict(hidden=hidden.contiguous(), hash_ids=ids.contiguous(), token_mask=mask)


def make_all(wl: Workload, device="cpu", T: int | None = None):
    d = dict(table=make_table(wl, device), table_scale=make_table_scale(wl, device))
    d.update(make_weights(wl, device))
    d.update(make_step_inputs(wl, device, T))
    d["row_offset"] = row_offsets(wl.rows)
    d["rows"] = np.asarray(wl.rows, np.int64)
    return d


def bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy of a tensor's raw bits (bf16 -> uint16, bytes -> uint8)."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype in (torch.uint8, torch.bool):
        return t.to(torch.uint8).cpu().numpy()
    return t.cpu().numpy()


def host_memory_bytes():
    """Memory this process may still pin on the host (cgroup limit aware)."""
    avail = None
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    try:
        lim = open("/sys/fs/cgroup/memory.max").read().strip()
        use = int(open("/sys/fs/cgroup/memory.current").read().strip())
        if lim != "max":
            cg = int(lim) - use
            avail = cg if avail is None else min(avail, cg)
    except (OSError, ValueError):
        pass
    return avail
