"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- a library conversion or matmul, a closed form, an
invariant the Engram pages state, or brute force on tiny inputs."""
import math

import numpy as np
import pytest
sympy = pytest.importorskip("sympy")
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.timeout(600) if hasattr(pytest.mark, "timeout") else []


def np_bf16(bits):
    """numpy's own widening of bf16 bit patterns (library route)."""
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_of(x_f32):
    return torch.from_numpy(np.asarray(x_f32, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_bf16_decode_all_patterns():
    b = np.arange(65536, dtype=np.uint16)
    ours = oracle.bf16_to_f64(b)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decode_all_codes():
    c = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(c)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert oracle.e4m3_to_f64(np.uint8(0x7E)) == 448.0
    assert oracle.e4m3_to_f64(np.uint8(0x01)) == 2.0 ** -9


def test_e8m0_decode():
    b = np.arange(255, dtype=np.uint8)
    ours = oracle.e8m0_to_f64(b)
    assert all(ours[i] == math.ldexp(1.0, i - 127) for i in range(255))
    assert np.isnan(oracle.e8m0_to_f64(np.uint8(255)))


def test_e4m3_encode_matches_torch_and_ties():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(4000) * 50,
        rng.standard_normal(2000) * 1e-2,
        rng.uniform(-463, 463, 2000),
    ])
    # exact midpoints between neighbouring finite codes (ties go to even)
    grid = np.sort(torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn)
                   .to(torch.float64).numpy())
    mids = (grid[1:] + grid[:-1]) / 2
    vals = np.concatenate([vals, mids, -mids, [0.0, -0.0, 448.0, -448.0, 450.0]])
    ours = oracle.f64_to_e4m3(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # saturation beyond the largest finite code
    assert oracle.f64_to_e4m3(np.array([1e4, -600.0, 480.0])).tolist() == [0x7E, 0xFE, 0x7E]


def test_bf16_round_matches_torch_and_ties():
    rng = np.random.default_rng(1)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-38).astype(np.float32)])
    ours = oracle.f64_to_bf16(f.astype(np.float64))
    assert np.array_equal(ours, bf16_bits_of(f))
    # exact ties in double between adjacent bf16 values: round to the even one
    lo = np.array([0x3F80, 0x3F81, 0xBF82, 0x4123], np.uint16)
    a, b = np_bf16(lo), np_bf16(lo + 1)
    mid = (a + b) / 2
    exp = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(mid), exp)
    # just past a tie (in magnitude) rounds away, even when binary32 would
    # lose the excess
    above = mid + mid * 2.0 ** -40
    assert np.array_equal(oracle.f64_to_bf16(above), (lo + 1).astype(np.uint16))


# --------------------------------------------------------------------------
# EngramLayout
# --------------------------------------------------------------------------

def test_layout_matches_consecutive_primes():
    for vocab, expect in ((2 ** 19, W.PRIMES_2POW19), (2 ** 23, W.PRIMES_2POW23)):
        primes, offsets = oracle.layout(vocab, 3, 8)
        ref = list(sympy.primerange(vocab, vocab + 4000))[:16]
        assert primes[0].tolist() == ref == list(expect)
        assert offsets[0].tolist() == [0] + np.cumsum(ref)[:-1].tolist()


def test_layout_multi_layer_primes_distinct_and_minimal():
    primes, offsets = oracle.layout(1000, 4, 3, n_layers=3)
    flat = primes.ravel().tolist()
    assert len(set(flat)) == len(flat) and all(sympy.isprime(p) for p in flat)
    # the union over layers is exactly the first len(flat) primes >= vocab
    assert sorted(flat) == list(sympy.primerange(1000, 2000))[:len(flat)]
    for l in range(3):
        assert offsets[l].tolist() == [0] + np.cumsum(primes[l])[:-1].tolist()


def test_tiny_rows_are_primes_in_range():
    assert all(sympy.isprime(p) for p in W.TINY_ROWS)
    assert min(W.TINY_ROWS) == 1009 and max(W.TINY_ROWS) == 1103


# --------------------------------------------------------------------------
# gather
# --------------------------------------------------------------------------

def test_gather_matches_direct_indexing_with_stride_and_bad_ids():
    rng = np.random.default_rng(2)
    rows = np.array([7, 11, 13, 17], np.int64)
    E = 8
    table = rng.integers(0, 65536, (rows.sum(), E), dtype=np.uint16)
    off = W.row_offsets(rows)
    ids_full = np.stack([rng.integers(0, r, 9) for r in rows], 1).astype(np.int32)
    ids_full = np.concatenate([ids_full, np.full((9, 3), -5, np.int32)], 1)  # padding cols
    ids = ids_full[:, :4]  # row stride 7 > C
    out, bad = oracle.gather(table, off, rows, ids, E)
    assert bad == 0
    assert np.array_equal(out, table[off[None, :] + ids])
    ids2 = ids.copy()
    ids2[3, 1] = 11       # == rows[1]: out of range
    ids2[5, 2] = -1
    out2, bad2 = oracle.gather(table, off, rows, ids2, E)
    assert bad2 == 2
    assert not out2[3, 1].any() and not out2[5, 2].any()
    assert np.array_equal(out2[0], out[0])


# --------------------------------------------------------------------------
# wkv
# --------------------------------------------------------------------------

def test_wkv_bf16_matches_numpy_matmul():
    rng = np.random.default_rng(3)
    A = bf16_bits_of(rng.standard_normal((5, 96)))
    Wt = bf16_bits_of(rng.standard_normal((40, 96)))
    kv = oracle.wkv_bf16(A, Wt)
    ref = np_bf16(A) @ np_bf16(Wt).T
    assert np.allclose(kv, ref, rtol=1e-12, atol=1e-12)


def test_wkv_mxfp8_matches_numpy_matmul():
    rng = np.random.default_rng(4)
    N, K = 64, 96
    A = bf16_bits_of(rng.standard_normal((3, K)) * 0.02)
    Wq = torch.from_numpy(rng.standard_normal((N, K))).to(torch.float8_e4m3fn)
    Ws = rng.integers(119, 128, (N // 32, K // 32)).astype(np.uint8)
    Wf = Wq.to(torch.float64).numpy() * np.ldexp(1.0, np.repeat(np.repeat(
        Ws.astype(np.int64) - 127, 32, 0), 32, 1))
    kv = oracle.wkv_mxfp8(A, Wq.view(torch.uint8).numpy(), Ws)
    assert np.allclose(kv, np_bf16(A) @ Wf.T, rtol=1e-12, atol=1e-15)


def _mx_qact_case(seed=14, T=5, K=128, N=96):
    """Random e4m3 codes for both operands (torch casts of normals: never a
    NaN code), activation scales that differ per token and per 32-k block,
    weight scales that differ per 32-row and per 32-k block, and the
    products decoded independently of the oracle: torch's float8_e4m3fn
    widening times an exact ldexp power of two."""
    rng = np.random.default_rng(seed)
    Aq = torch.from_numpy(rng.standard_normal((T, K)) * 40).to(torch.float8_e4m3fn)
    Wq = torch.from_numpy(rng.standard_normal((N, K))).to(torch.float8_e4m3fn)
    As = rng.permutation(np.arange(100, 100 + T * (K // 32))).reshape(T, K // 32).astype(np.uint8)
    Ws = rng.permutation(np.arange(112, 112 + (N // 32) * (K // 32))).reshape(
        N // 32, K // 32).astype(np.uint8)
    a_dec = Aq.to(torch.float64).numpy() * np.ldexp(1.0, np.repeat(As.astype(np.int64) - 127, 32, 1))
    w_dec = Wq.to(torch.float64).numpy() * np.ldexp(1.0, np.repeat(np.repeat(
        Ws.astype(np.int64) - 127, 32, 0), 32, 1))
    return (Aq.view(torch.uint8).numpy(), As, Wq.view(torch.uint8).numpy(), Ws,
            a_dec @ w_dec.T)


def test_wkv_mxfp8_qact_matches_numpy_matmul():
    """Both operands MXFP8 (the quantised-activation reference of the
    block-scaled MMA path): kv[t, n] = sum_k a(t, k) w(n, k), a with the
    scale of (token t, k-block k/32), w with that of (row block n/32,
    k-block k/32)."""
    Aq, As, Wq, Ws, ref = _mx_qact_case()
    kv = oracle.wkv_mxfp8_qact(Aq, As, Wq, Ws)
    assert kv.shape == ref.shape
    assert np.allclose(kv, ref, rtol=1e-12, atol=0.0)
    # a scale read with the wrong index would move whole 32-blocks by powers
    # of two: the check above is far tighter than that
    assert np.abs(ref).max() > 0


def test_forward_quantize_act_uses_quantised_rows_and_dequantised_weights():
    """forward(..., quantize_act=True) = mx_quantize (pinned above) of the
    gathered rows, then the contraction against the dequantised weights,
    recomputed here with torch and numpy."""
    wl = W.TINY_MXFP8
    d = W.make_all(wl, "cpu")
    Wq = W.bits(d["wkv"])
    Ws = d["wkv_scale"].numpy() if hasattr(d["wkv_scale"], "numpy") else d["wkv_scale"]
    r = oracle.forward(W.bits(d["table"]), d["row_offset"], d["rows"], d["hash_ids"].numpy(),
                       wl.head_dim, Wq, W.bits(d["hidden"]), W.bits(d["q_weight"]),
                       W.bits(d["k_weight"]), W.bits(d["token_mask"]), Ws=Ws,
                       quantize_act=True)
    T, K = wl.T, wl.K
    codes, scales = oracle.mx_quantize(r["rows"].reshape(T, K))
    a_dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * \
        np.ldexp(1.0, np.repeat(scales.astype(np.int64) - 127, 32, 1))
    w_dec = torch.from_numpy(np.ascontiguousarray(Wq).view(np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy() * np.ldexp(1.0, np.repeat(np.repeat(
            np.asarray(Ws).astype(np.int64) - 127, 32, 0), 32, 1))
    ref = a_dec @ w_dec.T
    assert np.allclose(r["kv"], ref, rtol=1e-12, atol=1e-300)
    # and it differs from the unquantised contraction (the rows really were quantised)
    plain = oracle.forward(W.bits(d["table"]), d["row_offset"], d["rows"],
                           d["hash_ids"].numpy(), wl.head_dim, Wq, W.bits(d["hidden"]),
                           W.bits(d["q_weight"]), W.bits(d["k_weight"]),
                           W.bits(d["token_mask"]), Ws=Ws)
    assert not np.array_equal(plain["kv"], r["kv"])


def test_mx_quantize_scale_is_minimal_and_codes_match_torch():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 128)) * np.array([1e-3, 0.02, 3.0, 700.0])[:, None]
    x[1, 32:64] = 0.0  # an all-zero block
    A = bf16_bits_of(x)
    codes, scales = oracle.mx_quantize(A)
    Af = np_bf16(A).reshape(4, 4, 32)
    e = scales.astype(np.int64) - 127
    amax = np.abs(Af).max(-1)
    nz = amax > 0
    assert np.all(amax[nz] <= 448.0 * np.ldexp(1.0, e[nz]))
    assert np.all(amax[nz] > 448.0 * np.ldexp(1.0, e[nz] - 1))
    assert e[1, 1] == 0 and not codes[1, 32:64].any()
    scaled = (Af * np.ldexp(1.0, -e)[..., None]).reshape(4, 128)
    ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


# --------------------------------------------------------------------------
# gate and residual: closed forms and invariants
# --------------------------------------------------------------------------

ONE = np.uint16(0x3F80)


def _identity_case(T=4, H=2, D=64, q=1.0, k=1.0, seed=6):
    """wkv maps the first D inputs straight to every key and to the value, so
    key_h = value = A[t, :D]; hidden[t, h] := A[t, :D]."""
    rng = np.random.default_rng(seed)
    K = D
    A = bf16_bits_of(rng.standard_normal((T, K)) * 0.3)
    Wt = np.zeros(((H + 1) * D, K), np.uint16)
    for blk in range(H + 1):
        Wt[blk * D + np.arange(D), np.arange(D)] = ONE
    kv = oracle.wkv_bf16(A, Wt)
    hidden = np.repeat(A[:, None, :D], H, 1)
    qb = np.full((H, D), bf16_bits_of(np.float32(q)), np.uint16)
    kb = np.full((H, D), bf16_bits_of(np.float32(k)), np.uint16)
    return A, kv, hidden, qb, kb


def test_gate_closed_form_identity_projection():
    for q, k in ((1.0, 1.0), (2.0, 0.5)):
        A, kv, hidden, qb, kb = _identity_case(q=q, k=k)
        T, H, D = hidden.shape
        eps = 1e-6
        r = oracle.gate(hidden, kv, qb, kb, None, eps=eps)
        m = (np_bf16(A) ** 2).mean(1)
        dot = math.sqrt(D) * m / (m + eps)
        assert np.allclose(r["dot"], dot[:, None], rtol=1e-12)
        g = 1.0 / (1.0 + np.exp(-np.sqrt(dot)))
        assert np.allclose(r["gate"], g[:, None], rtol=1e-12)
        exp_out = np_bf16(A)[:, None, :] * (1.0 + g[:, None, None])
        assert np.allclose(r["out_f64"], exp_out, rtol=1e-12)


def test_gate_q_zero_gives_sigmoid_of_clamp_root():
    A, kv, hidden, qb, kb = _identity_case()
    qb[:] = 0
    r = oracle.gate(hidden, kv, qb, kb, None)
    assert np.all(r["dot"] == 0.0)
    assert np.all(r["gate"] == 1.0 / (1.0 + math.exp(-math.sqrt(1e-6))))


def _random_case(T=6, H=3, D=128, seed=7):
    rng = np.random.default_rng(seed)
    hidden = bf16_bits_of(rng.standard_normal((T, H, D)))
    kv = rng.standard_normal((T, (H + 1) * D)) * 0.2
    qb = bf16_bits_of(rng.standard_normal((H, D)) * 0.5)
    kb = bf16_bits_of(rng.standard_normal((H, D)) * 0.5)
    return hidden, kv, qb, kb


def test_gate_sign_symmetry_and_range():
    hidden, kv, qb, kb = _random_case()
    r = oracle.gate(hidden, kv, qb, kb, None)
    r_neg = oracle.gate(hidden ^ np.uint16(0x8000), kv, qb, kb, None)
    assert np.allclose(r_neg["dot"], -r["dot"], rtol=1e-13)
    assert np.allclose(r_neg["gate"], 1.0 - r["gate"], rtol=1e-13)
    g = r["gate"]
    assert np.all((g > 0) & (g < 1))
    assert np.all(np.abs(g - 0.5) >= 1.0 / (1.0 + math.exp(-1e-3)) - 0.5 - 1e-15)


def test_gate_is_scale_invariant_in_hidden_and_key():
    hidden, kv, qb, kb = _random_case(D=64)
    T, H, D = hidden.shape
    r = oracle.gate(hidden, kv, qb, kb, None, eps=0.0)
    h2 = bf16_bits_of(np_bf16(hidden) * 4.0)  # exact power-of-two rescale
    kv2 = kv.copy()
    kv2[:, :H * D] *= 8.0
    r2 = oracle.gate(h2, kv2, qb, kb, None, eps=0.0)
    assert np.allclose(r2["dot"], r["dot"], rtol=1e-12)


def test_gate_value_shared_across_hc_copies():
    hidden, kv, qb, kb = _random_case()
    T, H, D = hidden.shape
    r = oracle.gate(hidden, kv, qb, kb, None)
    delta = (r["out_f64"] - np_bf16(hidden)) / r["gate"][:, :, None]
    value = kv[:, H * D:]
    assert np.allclose(delta, value[:, None, :], rtol=1e-9, atol=1e-12)


def test_gate_all_false_mask_passes_hidden_bits_through():
    hidden, kv, qb, kb = _random_case()
    hidden[0, 0, :4] = [0x8000, 0x7F80, 0xFF80, 0x0001]  # -0, +inf, -inf, subnormal
    mask = np.zeros(hidden.shape[0], np.uint8)
    r = oracle.gate(hidden, kv, qb, kb, mask)
    assert np.array_equal(r["out_bf16"], hidden)
    assert np.all(r["gate"] == 0.0)
    mask[2] = 1
    r2 = oracle.gate(hidden, kv, qb, kb, mask)
    assert not np.array_equal(r2["out_bf16"][2], hidden[2])
    assert np.array_equal(r2["out_bf16"][3], hidden[3])


def test_gate_strided_hidden_matches_contiguous():
    hidden, kv, qb, kb = _random_case()
    big = np.zeros((hidden.shape[0], hidden.shape[1] + 2, hidden.shape[2] * 2), np.uint16)
    big[:, 1:-1, ::2] = hidden
    r = oracle.gate(hidden, kv, qb, kb, None)
    r2 = oracle.gate(big[:, 1:-1, ::2], kv, qb, kb, None)
    assert np.array_equal(r["out_bf16"], r2["out_bf16"])


def test_forward_tiny_end_to_end_composition():
    wl = W.TINY
    d = W.make_all(wl, "cpu")
    r = oracle.forward(W.bits(d["table"]), d["row_offset"], d["rows"],
                       d["hash_ids"].numpy(), wl.head_dim, W.bits(d["wkv"]),
                       W.bits(d["hidden"]), W.bits(d["q_weight"]), W.bits(d["k_weight"]),
                       W.bits(d["token_mask"]))
    T, C, E = wl.T, wl.n_hash_cols, wl.head_dim
    assert r["n_bad"] == 0
    table = W.bits(d["table"])
    ids = d["hash_ids"].numpy()
    assert np.array_equal(r["rows"], table[d["row_offset"][None, :] + ids])
    kv = np_bf16(r["rows"].reshape(T, C * E)) @ np_bf16(W.bits(d["wkv"])).T
    assert np.allclose(r["kv"], kv, rtol=1e-10, atol=1e-12)
    mask = W.bits(d["token_mask"]).astype(bool)
    assert 0 < mask.sum() < T
    assert np.array_equal(r["out_bf16"][~mask], W.bits(d["hidden"])[~mask])


def test_gather_e4m3_table_matches_torch_dequant_and_indexing():
    """fp8 table rows (class ParallelEngramEmbedding: e4m3 with one ue8m0 scale
    per 32 elements, dequantized to bf16 on lookup) against torch's own
    float8_e4m3fn -> float64 decode, an exact power-of-two scaling, and its
    RTNE cast to bfloat16; plus direct row indexing and bad ids."""
    E = 64
    scale_bytes = [0, 1, 9, 60, 113, 118, 121, 127, 128, 140, 200, 253, 254]
    # every code appears in each block position, under every scale byte
    codes = np.tile(np.arange(256, dtype=np.uint8).reshape(4, 64), (len(scale_bytes), 1))
    scales = np.repeat(np.array(scale_bytes, np.uint8), 4)[:, None].repeat(2, axis=1).copy()
    scales[::2, 1] = 127  # a second block with another scale in half of the rows
    n = codes.shape[0]
    rows = np.array([n], np.int64)
    ids = np.arange(n, dtype=np.int32).reshape(-1, 1)
    got, bad = oracle.gather_e4m3(codes, scales, [0], rows, ids, E)
    assert bad == 0
    dq = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    mult = torch.from_numpy(np.ldexp(1.0, scales.astype(np.int64) - 127))  # exact
    ref = (dq * mult.repeat_interleave(32, dim=1)).to(torch.bfloat16).view(torch.int16)
    ref = ref.numpy().view(np.uint16)
    g = got[:, 0, :]
    refnan = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x7F) != 0)
    gotnan = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    assert np.array_equal(refnan, gotnan)          # the NaN codes S.1111.111
    assert refnan.sum() == 2 * len(scale_bytes)    # (0x7F and 0xFF once per scale byte)
    assert np.array_equal(g[~refnan], ref[~refnan])

    # rows by direct indexing: strided ids, per-column offsets, bad ids
    rng = np.random.default_rng(5)
    rws = np.array([7, 11, 13], np.int64)
    off = W.row_offsets(rws)
    tc = rng.integers(0, 256, (rws.sum(), E), dtype=np.uint8)
    ts = rng.integers(110, 130, (rws.sum(), E // 32), dtype=np.uint8)
    full = np.stack([rng.integers(0, r, 6) for r in rws], 1).astype(np.int32)
    full = np.concatenate([full, np.full((6, 2), -9, np.int32)], 1)
    idv = full[:, :3]                               # row stride 5 > C
    out, bad = oracle.gather_e4m3(tc, ts, off, rws, idv, E)
    assert bad == 0
    one, _ = oracle.gather_e4m3(tc, ts, [0], [rws.sum()], (off[None, :] + idv).reshape(-1, 1)
                                .astype(np.int32), E)
    assert np.array_equal(out.reshape(-1, E), one[:, 0, :])
    idv2 = idv.copy()
    idv2[1, 2] = 13      # == rows[2]
    idv2[4, 0] = -1
    out2, bad2 = oracle.gather_e4m3(tc, ts, off, rws, idv2, E)
    assert bad2 == 2 and not out2[1, 2].any() and not out2[4, 0].any()
    assert np.array_equal(out2[0], out[0])
