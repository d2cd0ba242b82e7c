"""The synthetic inputs follow their stated recipe: configuration shapes,
prime row counts, value distributions, id and mask distributions, code and
scale ranges, and determinism under a seed.  Sized to run in seconds."""
import dataclasses

import numpy as np
import pytest
sympy = pytest.importorskip("sympy")
import torch

import workloads as W


def _f32(t):
    return t.float().numpy().astype(np.float64)


def test_configuration_shapes():
    # (T, dim, hc_mult, n_hash_cols, head_dim, K, N)
    want = {"tiny": (16, 256, 2, 8, 32, 256, 768),
            "decode": (64, 4096, 4, 16, 64, 1024, 20480),
            "prefill": (8192, 4096, 4, 16, 64, 1024, 20480),
            "offload": (256, 4096, 4, 16, 64, 1024, 20480)}
    for name, shape in want.items():
        wl = W.ALL[name]
        assert (wl.T, wl.dim, wl.hc_mult, wl.n_hash_cols, wl.head_dim, wl.K, wl.N) == shape
    for wl in (W.MXFP8_DECODE, W.MXFP8_PREFILL):
        assert (wl.dim, wl.N, wl.K, wl.wkv_format) == (7168, 35840, 1024, "mxfp8")
    assert (W.MXFP8_DECODE.T, W.MXFP8_PREFILL.T) == (64, 4096)
    assert len({wl.seed for wl in W.ALL.values()}) == len(W.ALL)


def test_row_counts_are_the_layout_primes():
    # decode-shaped tables: the 16 consecutive primes above 2^19 - 1
    p, out = [], 2 ** 19 - 1
    for _ in range(16):
        out = sympy.nextprime(out)
        p.append(out)
    assert list(W.DECODE.rows) == p and W.DECODE.total_rows == sum(p)
    q, out = [], 2 ** 23 - 1
    for _ in range(16):
        out = sympy.nextprime(out)
        q.append(out)
    assert list(W.OFFLOAD.rows) == q
    assert all(sympy.isprime(r) for r in W.TINY.rows) and len(W.TINY.rows) == 8
    assert np.array_equal(W.row_offsets([3, 5, 7]), [0, 3, 8])


def test_weight_and_hidden_distributions():
    w = W.make_weights(W.DECODE)
    x = _f32(w["wkv"])
    assert x.shape == (20480, 1024) and w["wkv"].dtype == torch.bfloat16
    assert abs(x.mean()) < 1e-4 and abs(x.std() / 0.02 - 1) < 0.01
    for k in ("q_weight", "k_weight"):
        assert w[k].shape == (4, 4096) and abs(_f32(w[k]).std() / 0.02 - 1) < 0.05
    h = _f32(W.make_step_inputs(W.DECODE)["hidden"])
    assert h.shape == (64, 4, 4096) and abs(h.std() - 1) < 0.01 and abs(h.mean()) < 0.01
    t = _f32(W.make_table(W.TINY))
    assert t.shape == (sum(W.TINY.rows), 32) and abs(t.std() / 0.02 - 1) < 0.03


def test_mxfp8_codes_and_scales():
    w = W.make_weights(W.TINY_MXFP8)
    codes, sc = w["wkv"].numpy(), w["wkv_scale"].numpy()
    N, K = W.TINY_MXFP8.N, W.TINY_MXFP8.K
    assert codes.shape == (N, K) and sc.shape == (N // 32, K // 32)
    assert sc.min() >= 119 and sc.max() <= 127 and len(np.unique(sc)) == 9
    assert not np.any((codes & 0x7F) == 0x7F)  # no NaN code
    # the codes are the e4m3 rounding of N(0, 1): about 68 % within magnitude 1
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert abs(np.mean(np.abs(v) <= 1.0) - 0.683) < 0.03


def test_fp8_table_codes_and_scales():
    wl = W.TINY_E4M3
    codes, sc = W.make_table(wl), W.make_table_scale(wl)
    assert codes.dtype == torch.uint8 and codes.shape == (wl.total_rows, wl.head_dim)
    assert sc.shape == (wl.total_rows, wl.head_dim // 32)
    s = sc.numpy()
    assert s.min() >= 113 and s.max() <= 121 and len(np.unique(s)) == 9
    assert not np.any((codes.numpy() & 0x7F) == 0x7F)
    assert W.make_table_scale(W.TINY) is None


def test_uniform_ids_and_mask_rate():
    wl = W.TINY
    T = 40000
    st = W.make_step_inputs(wl, T=T)
    ids = st["hash_ids"].numpy()
    rows = np.asarray(wl.rows)
    assert ids.shape == (T, 8) and ids.dtype == np.int32
    assert np.all(ids >= 0) and np.all(ids < rows)
    # uniform: the mean of id / rows is 1/2 within a few standard errors
    u = (ids + 0.5) / rows
    assert np.all(np.abs(u.mean(axis=0) - 0.5) < 4 * np.sqrt(1 / 12 / T))
    m = st["token_mask"].numpy()
    assert abs(m.mean() - 0.75) < 0.01
    pre = dataclasses.replace(W.PREFILL, dim=256)
    assert abs(W.make_step_inputs(pre, T=T)["token_mask"].numpy().mean() - 0.9) < 0.01
    assert W.make_step_inputs(W.DECODE)["token_mask"] is None


def test_zipf_ids_are_scattered_zipf():
    rows = list(W.PREFILL.rows[:2])
    T = 40000
    ids = W._zipf_ids(rows, T, np.random.default_rng(7))
    for c, p in enumerate(rows):
        col = ids[:, c]
        assert np.all((col >= 0) & (col < p))
        vals, counts = np.unique(col, return_counts=True)
        # rank 0 lands on row b = (7919 (c + 1) + 13) mod p, with probability
        # 1 / sum_{r=1..p} r^-1.1
        z = float(np.sum(np.arange(1, p + 1, dtype=np.float64) ** -1.1))
        top = vals[np.argmax(counts)]
        assert top == (7919 * (c + 1) + 13) % p
        assert abs(counts.max() / T - 1 / z) < 0.01
        # rank 1 is the next most frequent: 2^-1.1 of rank 0
        a = (2654435761 % p) or 1
        assert counts[vals == (a + (7919 * (c + 1) + 13)) % p][0] / counts.max() == \
            pytest.approx(2 ** -1.1, abs=0.08)


def test_seeded_inputs_are_deterministic():
    a, b = W.make_all(W.TINY), W.make_all(W.TINY)
    for k in ("table", "wkv", "q_weight", "k_weight", "hidden", "hash_ids", "token_mask"):
        assert torch.equal(a[k], b[k]), k
    c = W.make_step_inputs(W.TINY, step=1)
    assert not torch.equal(a["hidden"], c["hidden"])
