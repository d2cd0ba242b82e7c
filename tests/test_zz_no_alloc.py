"""engram_gate_noalloc: the gate and masked residual over a kv projection
the caller computed, with its cross-CTA partial sums in a fixed device
array instead of allocated memory.

Its output is checked against the oracle's gate and residual on the same
bf16 kv, and against engram_forward (the handle's own path) on the same
inputs, for two calls in a row with different inputs and sizes, so a call
that read another call's leftover partials would fail.  The file sorts
after the single-layer parity files, so it also runs once those have used
the device; it builds its own layers and passes alone as well."""
import numpy as np
import pytest
import torch

import workloads as W
from engram_case import Case, np_bf16
from hashed_gram_engram_gb300 import EngramError, _lib

MAX = _lib.ENGRAM_NOALLOC_MAX_PARTIALS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _strides(x):
    return tuple(x.stride())


def _noalloc(case, inp, kv, out=None):
    hidden = inp["hidden"]
    T, H, D = hidden.shape
    out = torch.empty_like(hidden) if out is None else out
    _lib.engram_gate_noalloc(hidden, _strides(hidden), kv, kv.stride(0), case.q, case.k,
                             inp["token_mask"], out, _strides(out), T, H, D,
                             eps=case.wl.eps, clamp=case.wl.clamp,
                             stream=torch.cuda.current_stream())
    return out


def _kv(case, T):
    """kv = rows . wkv^T from the rows the handle staged, rounded to bf16
    (what a caller's own bf16 GEMM hands over)."""
    rows = case.layer.staged_rows(T)
    return (rows.float() @ case.wkv.float().t()).to(torch.bfloat16)


def _check(case, inp, got, ref, kv):
    """Rounding-level agreement with engram_forward: the two differ by the
    bf16 rounding of kv (keys and value) and the final bf16 rounding of
    each output."""
    H, D = case.wl.hc_mult, case.wl.dim
    a = np_bf16(W.bits(got))
    b = np_bf16(W.bits(ref))
    v = np_bf16(W.bits(kv[:, H * D:]))[:, None, :]
    bound = 2.0 ** -7 * np.abs(b) + 2.0 ** -7 * np.abs(v) + 1e-5
    assert np.all(np.abs(a - b) <= bound), f"max diff {np.abs(a - b).max()}"
    if inp["token_mask"] is not None:
        m = W.bits(inp["token_mask"]).astype(bool)
        assert np.array_equal(W.bits(got)[~m], W.bits(inp["hidden"])[~m])


def test_sizes_beyond_scratch_are_refused():
    # Fake, aligned, non-overlapping addresses: the size checks come before
    # any CUDA call, so nothing is dereferenced and no device is needed.
    T, H, D = MAX // 4 + 1, 4, 256
    base = 1 << 40
    hid, out, kv, q, k = (base + i * (1 << 36) for i in range(5))
    st = (H * D, D, 1)
    with pytest.raises(EngramError) as e:
        _lib.engram_gate_noalloc(hid, st, kv, (H + 1) * D, q, k, None, out, st, T, H, D)
    assert e.value.code == _lib.ENGRAM_ERR_SCRATCH_LIMIT
    # T * H * (D / 256) over the limit through D as well
    with pytest.raises(EngramError) as e:
        _lib.engram_gate_noalloc(hid, (4 * 8192, 8192, 1), kv, 5 * 8192, q, k, None, out,
                                 (4 * 8192, 8192, 1), MAX // 128 + 1, 4, 8192)
    assert e.value.code == _lib.ENGRAM_ERR_SCRATCH_LIMIT
    with pytest.raises(EngramError) as e:
        _lib.engram_gate_noalloc(hid, st, kv, (H + 1) * D, q, k, None, out, st, 4, 5, D)
    assert e.value.code == _lib.ENGRAM_ERR_INVALID_ARG


@pytest.mark.gpu
def test_two_calls_match_engram_forward():
    for wl, sizes in ((W.DECODE, (64, 17)), (W.TINY, (1000, 3))):
        case = Case(wl, max_tokens=max(sizes))
        _lib.engram_gate_noalloc(None, None, None, 0, None, None, None, None, None, 0,
                                 wl.hc_mult, wl.dim)  # per-device setup, launches nothing
        calls = []
        for step, T in enumerate(sizes):
            inp = case.step_inputs(T=T, step=100 + step)
            ref = case.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
            kv = _kv(case, T)
            out = torch.empty_like(inp["hidden"])
            calls.append((inp, ref, kv, out))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for inp, ref, kv, out in calls:  # two calls in a row
            _noalloc(case, inp, kv, out)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across the calls"
        for inp, ref, kv, out in calls:
            _check(case, inp, out, ref, kv)
        # run to run the same bits
        inp, ref, kv, out = calls[0]
        again = _noalloc(case, inp, kv)
        torch.cuda.synchronize()
        assert torch.equal(again, out)
        case.layer.close()


@pytest.mark.gpu
def test_matches_oracle_gate_on_the_same_kv():
    """Against the oracle's gate and residual (fp64) on the very bf16 kv the
    entry point is given, widened exactly: the only differences left are the
    kernel's fp32 sums and the final bf16 rounding of each output."""
    import oracle
    for wl, T in ((W.DECODE, 64), (W.TINY, 333)):
        case = Case(wl, max_tokens=T)
        inp = case.step_inputs(T=T, step=300)
        case.layer.lookup(inp["hash_ids"])
        kv = _kv(case, T)
        out = _noalloc(case, inp, kv)
        torch.cuda.synchronize()
        mask = None if inp["token_mask"] is None else W.bits(inp["token_mask"])
        ref = oracle.gate(W.bits(inp["hidden"]), np_bf16(W.bits(kv)), W.bits(case.q),
                          W.bits(case.k), mask, wl.eps, wl.clamp)
        got = np_bf16(W.bits(out))
        exp = ref["out_f64"]
        v = np_bf16(W.bits(kv[:, wl.hc_mult * wl.dim:]))[:, None, :]
        bound = 2.0 ** -8 * np.abs(exp) + 1e-5 * np.abs(v) + 1e-6
        assert np.all(np.abs(got - exp) <= bound), f"max diff {np.abs(got - exp).max()}"
        assert np.abs(got - exp).max() <= wl.tol
        if mask is not None:
            m = mask.astype(bool)
            assert np.array_equal(W.bits(out)[~m], W.bits(inp["hidden"])[~m])
        case.layer.close()


@pytest.mark.gpu
def test_in_place_and_largest_size():
    wl = W.TINY  # H = 2, D = 256: one slot per (token, copy)
    T = MAX // wl.hc_mult
    case = Case(wl, max_tokens=T)
    inp = case.step_inputs(T=T, step=7)
    ref = case.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
    kv = _kv(case, T)
    work = inp["hidden"].clone()
    _lib.engram_gate_noalloc(work, _strides(work), kv, kv.stride(0), case.q, case.k,
                             inp["token_mask"], work, _strides(work), T, wl.hc_mult, wl.dim,
                             eps=wl.eps, clamp=wl.clamp, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    _check(case, inp, work, ref, kv)
    with pytest.raises(EngramError) as e:
        _noalloc(case, case.step_inputs(T=T + 1, step=8), kv)
    assert e.value.code == _lib.ENGRAM_ERR_SCRATCH_LIMIT
    case.layer.close()
