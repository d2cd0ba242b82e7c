"""GPU parity: the CUDA path through the C ABI against the oracle.

Element-by-element on sizes the oracle finishes in seconds (several tiles
and ragged tails on both wkv schedules), whole-output at the decode
config, every token of the prefill config (the oracle spread over the
host's cores), plus the edge cases: T = 0, maximum T (also with an odd
number of 128-token tiles, where the GEMM's last CTA pair reads padding),
all-False masks, in-place and strided views, out-of-range ids, and
run-to-run determinism."""

import numpy as np
import pytest
import torch

import workloads as W
from engram_case import Case, compare, oracle_all
from hashed_gram_engram_gb300 import EngramError, ENGRAM_DEVERR_BAD_HASH_ID

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.fixture(scope="module")
def tiny():
    return Case(W.TINY, max_tokens=1024)


def _run(case, inp, T=None):
    out = case.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    T = inp["hidden"].shape[0] if T is None else T
    gate, value = case.layer.intermediates(T)
    torch.cuda.synchronize()
    return out, gate, value


def test_tiny_forward_matches_oracle(tiny):
    inp = tiny.step_inputs()
    out, gate, value = _run(tiny, inp)
    ref = tiny.oracle(inp)
    compare(tiny, inp, out, ref, gate=gate, value=value)
    # the gather is bit-exact
    rows = tiny.layer.staged_rows(W.TINY.T)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(rows), ref["rows"].reshape(W.TINY.T, -1))
    assert tiny.layer.device_error() == 0


@pytest.mark.parametrize("T", [1, 5, 16, 31, 100, 255, 256])
def test_tokens_as_n_path_ragged_T(tiny, T):
    inp = tiny.step_inputs(T=T, step=T)
    out, gate, value = _run(tiny, inp)
    compare(tiny, inp, out, tiny.oracle(inp), gate=gate, value=value)


@pytest.mark.parametrize("T", [257, 300, 640, 1024])
def test_tokens_as_m_path_ragged_T(tiny, T):
    inp = tiny.step_inputs(T=T, step=T)
    out, gate, value = _run(tiny, inp)
    compare(tiny, inp, out, tiny.oracle(inp), gate=gate, value=value)


@pytest.mark.parametrize("T", [300, 600])
def test_max_tokens_with_odd_token_tiles(T):
    """T = max_tokens with 3 or 5 tiles of 128 tokens: the prefill GEMM's CTA
    pairs take tiles 2i and 2i + 1, so the last pair's second tile lies past
    T, in the staging buffer's padding (max_tokens rounded up to 256); its
    rows must leave no trace in the output."""
    case = Case(W.TINY, max_tokens=T)
    inp = case.step_inputs(T=T, step=T + 11)
    out, gate, value = _run(case, inp)
    compare(case, inp, out, case.oracle(inp), gate=gate, value=value)
    case.layer.close()


def test_separate_lookup_then_forward(tiny):
    inp = tiny.step_inputs(T=40, step=7)
    tiny.layer.lookup(inp["hash_ids"])
    out = tiny.layer.forward(inp["hidden"], None, inp["token_mask"])
    torch.cuda.synchronize()
    compare(tiny, inp, out, tiny.oracle(inp))


def test_background_lookup_matches(tiny):
    inp = tiny.step_inputs(T=300, step=8)
    tiny.layer.lookup(inp["hash_ids"], background=True)
    out = tiny.layer.forward(inp["hidden"], None, inp["token_mask"])
    torch.cuda.synchronize()
    compare(tiny, inp, out, tiny.oracle(inp))


def test_all_false_mask_passes_hidden_through(tiny):
    for T in (16, 300):
        inp = tiny.step_inputs(T=T, step=9)
        inp["token_mask"] = torch.zeros(T, dtype=torch.uint8, device="cuda")
        h = inp["hidden"]
        h[0, 0, :4] = torch.tensor([-0.0, float("inf"), float("-inf"), 1e-40],
                                   dtype=torch.bfloat16)
        out, gate, _ = _run(tiny, inp)
        assert torch.equal(out.view(torch.int16), h.view(torch.int16))
        assert torch.all(gate == 0)


def test_gate_range_and_shared_value(tiny):
    inp = tiny.step_inputs(T=64, step=10)
    inp["token_mask"] = None
    out, gate, value = _run(tiny, inp)
    g = gate.double().cpu().numpy()
    assert np.all((g > 0) & (g < 1)) and np.all(np.abs(g - 0.5) >= 2.4e-4)


def test_in_place_and_strided_views(tiny):
    T = 48
    inp = tiny.step_inputs(T=T, step=11)
    ref = tiny.oracle(inp)
    H, D = W.TINY.hc_mult, W.TINY.dim
    # strided: hc copies padded apart, tokens padded apart
    big = torch.zeros((T, H + 1, D + 64), dtype=torch.bfloat16, device="cuda")
    big[:, :H, :D] = inp["hidden"]
    hv = big[:, :H, :D]
    outbig = torch.full((T, H, D + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    ov = outbig[:, :, :D]
    tiny.layer.forward(hv, inp["hash_ids"], inp["token_mask"], out=ov)
    torch.cuda.synchronize()
    compare(tiny, inp, ov, ref)
    assert torch.all(outbig[:, :, D:] == 7.0)
    # in place
    h2 = inp["hidden"].clone()
    tiny.layer.forward(h2, inp["hash_ids"], inp["token_mask"], out=h2)
    torch.cuda.synchronize()
    assert torch.equal(h2.view(torch.int16), ov.contiguous().view(torch.int16))


def test_prefill_path_views(tiny):
    """The prefill kernels (T > 256) on strided, broadcast and in-place views:
    padded copies and tokens (hidden staged by TMA boxes), copies broadcast
    with a zero stride (a view TMA cannot describe: the GEMM's plain-load
    instance), and out = hidden."""
    T = 600
    inp = tiny.step_inputs(T=T, step=13)
    ref = tiny.oracle(inp)
    H, D = W.TINY.hc_mult, W.TINY.dim
    big = torch.zeros((T + 3, H + 1, D + 64), dtype=torch.bfloat16, device="cuda")
    big[:T, :H, :D] = inp["hidden"]
    hv = big[:T, :H, :D]
    out = tiny.layer.forward(hv, inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    compare(tiny, inp, out, ref, value_rtol=2.0 ** -8 + 1e-3)
    # copies broadcast from one row per token
    hb = inp["hidden"][:, 0, :].clone()[:, None, :].expand(T, H, D)
    assert hb.stride(1) == 0
    inp_b = dict(inp, hidden=hb)
    out_b = tiny.layer.forward(hb, inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    compare(tiny, inp_b, out_b, tiny.oracle(inp_b), value_rtol=2.0 ** -8 + 1e-3)
    # in place
    h2 = inp["hidden"].clone()
    tiny.layer.forward(h2, inp["hash_ids"], inp["token_mask"], out=h2)
    torch.cuda.synchronize()
    assert torch.equal(h2.view(torch.int16), out.view(torch.int16))
    assert tiny.layer.device_error() == 0


def test_strided_hash_ids(tiny):
    T = 70
    inp = tiny.step_inputs(T=T, step=12)
    wide = torch.full((T, W.TINY.n_hash_cols + 5), -1, dtype=torch.int32, device="cuda")
    wide[:, :W.TINY.n_hash_cols] = inp["hash_ids"]
    out = tiny.layer.forward(inp["hidden"], wide[:, :W.TINY.n_hash_cols], inp["token_mask"])
    torch.cuda.synchronize()
    compare(tiny, inp, out, tiny.oracle(inp))


def test_deterministic_across_runs(tiny):
    for T in (77, 513):
        inp = tiny.step_inputs(T=T, step=13)
        a = tiny.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
        b = tiny.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_zero_tokens_and_limits(tiny):
    empty_h = torch.empty((0, W.TINY.hc_mult, W.TINY.dim), dtype=torch.bfloat16, device="cuda")
    empty_ids = torch.empty((0, W.TINY.n_hash_cols), dtype=torch.int32, device="cuda")
    out = tiny.layer.forward(empty_h, empty_ids)
    assert out.shape == empty_h.shape
    tiny.layer.lookup(empty_ids)
    big = tiny.step_inputs(T=1025, step=14)
    with pytest.raises(EngramError) as e:
        tiny.layer.forward(big["hidden"], big["hash_ids"])
    assert e.value.code == -3
    inp = tiny.step_inputs(T=8, step=15)
    with pytest.raises(EngramError) as e:  # overlapping, non-identical out
        tiny.layer.forward(inp["hidden"][1:], inp["hash_ids"][1:], out=inp["hidden"][:-1])
    assert e.value.code == -1
    with pytest.raises(EngramError) as e:  # staged rows of another T
        tiny.layer.lookup(inp["hash_ids"][:4])
        tiny.layer.forward(inp["hidden"], None)
    assert e.value.code == -1
    torch.cuda.synchronize()
    assert tiny.layer.device_error() == 0


def test_out_of_range_ids_zero_the_row_and_flag(tiny):
    T = 20
    inp = tiny.step_inputs(T=T, step=16)
    ids = inp["hash_ids"].clone()
    ids[3, 2] = W.TINY.rows[2]  # one past the end
    ids[7, 5] = -4
    tiny.layer.forward(inp["hidden"], ids, inp["token_mask"])
    torch.cuda.synchronize()
    assert tiny.layer.device_error() & ENGRAM_DEVERR_BAD_HASH_ID
    rows = W.bits(tiny.layer.staged_rows(T)).reshape(T, W.TINY.n_hash_cols, W.TINY.head_dim)
    assert not rows[3, 2].any() and not rows[7, 5].any()
    assert tiny.layer.device_error() == 0  # cleared


# ---------------------------------------------------------------- full configs

@pytest.fixture(scope="module")
def decode():
    return Case(W.DECODE, max_tokens=W.PREFILL.T)


def test_decode_config_full(decode):
    inp = decode.step_inputs()
    out, gate, value = _run(decode, inp)
    ref = decode.oracle(inp)
    res = compare(decode, inp, out, ref, gate=gate, value=value)
    assert decode.layer.device_error() == 0
    print("decode", res)
    # the gather kernel (engram_lookup) is bit-exact on the full-size table, and
    # the forward that consumes its staged rows matches the forward that
    # gathers the rows itself bit for bit
    decode.layer.lookup(inp["hash_ids"])
    rows = decode.layer.staged_rows(W.DECODE.T)
    out2 = decode.layer.forward(inp["hidden"], None, inp["token_mask"])
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(rows), ref["rows"].reshape(W.DECODE.T, -1))
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("T", [1, 17, 100, 128, 129, 256])
def test_decode_shapes_ragged_T(decode, T):
    inp = decode.step_inputs(T=T, step=T)
    out, gate, value = _run(decode, inp)
    tokens = None if T <= 128 else np.unique(np.r_[0, 1, T // 2, T - 2, T - 1,
                                                   np.random.default_rng(T).choice(T, 12)])
    compare(decode, inp, out, decode.oracle(inp, tokens=tokens), tokens=tokens, gate=gate,
            value=value)


def test_decode_out_of_range_ids_read_zero_rows(decode):
    T = 32
    inp = decode.step_inputs(T=T, step=99)
    ids = inp["hash_ids"].clone()
    ids[3, 2] = W.DECODE.rows[2]
    ids[9, 15] = -7
    ids[31, 0] = 2 ** 31 - 1
    inp["hash_ids"] = ids
    out, gate, value = _run(decode, inp)
    ref = decode.oracle(inp)
    assert ref["n_bad"] == 3
    compare(decode, inp, out, ref, gate=gate, value=value)
    assert decode.layer.device_error() & ENGRAM_DEVERR_BAD_HASH_ID


def test_prefill_config_every_token(decode):
    """The prefill configuration (T = 8192, Zipf(1.1) ids, Bernoulli(0.9)
    mask) at every token: the staged rows bit for bit, the output, gate and
    value against the oracle run over the host's cores."""
    wl = W.PREFILL
    case = decode
    case.wl = wl  # same weights and table; prefill ids, mask and T
    try:
        inp = case.step_inputs()
        out, gate, value = _run(case, inp)
        rows = case.layer.staged_rows(wl.T)
        torch.cuda.synchronize()
        ref = oracle_all(case, inp)
        assert np.array_equal(W.bits(rows), ref["rows"].reshape(wl.T, -1))
        compare(case, inp, out, ref, gate=gate, value=value)
        m = W.bits(inp["token_mask"]).astype(bool)
        assert 0 < (~m).sum() < wl.T
        g = gate.double().cpu().numpy()
        assert np.all(g[~m] == 0) and np.all((g[m] > 0) & (g[m] < 1))
        assert case.layer.device_error() == 0
    finally:
        case.wl = W.DECODE


def test_graph_capture_replays_bit_identically(decode):
    """A captured forward replays to the same bits (the grid barrier resets itself)."""
    inp = decode.step_inputs(T=64, step=21)
    ref = decode.layer.forward(inp["hidden"], inp["hash_ids"], None)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = torch.empty_like(inp["hidden"])
    with torch.cuda.stream(s):
        decode.layer.forward(inp["hidden"], inp["hash_ids"], None, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        decode.layer.forward(inp["hidden"], inp["hash_ids"], None, out=out, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert decode.layer.device_error() == 0


def test_forward_host_buffers(tiny):
    inp = tiny.step_inputs(T=24, step=22)
    ref = tiny.oracle(inp)
    hid = inp["hidden"].cpu().pin_memory()
    ids = inp["hash_ids"].cpu().pin_memory()
    mask = inp["token_mask"].cpu().pin_memory()
    out = torch.empty_like(hid).pin_memory()
    tiny.layer.forward_host(hid, ids, mask, out)
    torch.cuda.synchronize()
    compare(tiny, inp, out, ref)
