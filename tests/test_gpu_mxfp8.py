"""GPU parity of the MXFP8 wkv path (e4m3 weights with E8M0 32 x 32 block
scales; the gathered rows quantised to e4m3 with one E8M0 scale per 32 k).

Three bars, from strictest:
  - the quantised activations (codes and scales) equal the oracle's
    quantisation of the gathered rows bit for bit;
  - the output matches the oracle run on those same quantised activations
    at rounding level, with gate and value within 1e-3 relative;
  - the output matches the plain oracle (unquantised activations, the
    layer's definition) within the configuration's tolerance, gate and
    value within 5e-2 relative.
Both schedules are covered: the fused decode kernel (T <= 128) and the
prefill tiles (T > 128)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from engram_case import Case, compare, oracle_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.fixture(scope="module")
def tiny_mx():
    return Case(W.TINY_MXFP8, max_tokens=1024)


@pytest.fixture(scope="module")
def mx():
    return Case(W.MXFP8_DECODE, max_tokens=W.MXFP8_PREFILL.T)


def _run(case, inp):
    out = case.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    gate, value = case.layer.intermediates(inp["hidden"].shape[0])
    torch.cuda.synchronize()
    return out, gate, value


def _check_all(case, inp, out, gate, value, tokens=None):
    T = inp["hidden"].shape[0]
    ref_q = case.oracle(inp, tokens=tokens, quantize_act=True)
    # the fused kernel keeps the value in fp32; the prefill tiles store it
    # as bf16, whose rounding alone is up to 2^-8 relative
    value_rtol = 1e-3 if T <= 128 else 2.0 ** -8 + 1e-3
    compare(case, inp, out, ref_q, tokens=tokens, gate=gate, value=value,
            value_rtol=value_rtol, gate_rtol=1e-3)
    ref = case.oracle(inp, tokens=tokens)
    compare(case, inp, out, ref, tokens=tokens, gate=gate, value=value, value_rtol=5e-2,
            gate_rtol=5e-2, rounding=False)
    # the activation quantisation is bit-exact
    codes, scales = case.layer.staged_mx(T)
    torch.cuda.synchronize()
    A = ref["rows"].reshape(ref["rows"].shape[0], -1)
    q_ref, s_ref = oracle.mx_quantize(A)
    sel = slice(None) if tokens is None else tokens
    assert np.array_equal(codes.cpu().numpy()[sel], q_ref)
    assert np.array_equal(scales.cpu().numpy()[sel], s_ref)
    assert case.layer.device_error() == 0


@pytest.mark.parametrize("T", [1, 16, 17, 100, 128])
def test_tiny_mxfp8_fused_path(tiny_mx, T):
    inp = tiny_mx.step_inputs(T=T, step=T)
    out, gate, value = _run(tiny_mx, inp)
    _check_all(tiny_mx, inp, out, gate, value)


@pytest.mark.parametrize("T", [129, 300, 1024])
def test_tiny_mxfp8_prefill_path(tiny_mx, T):
    inp = tiny_mx.step_inputs(T=T, step=T)
    out, gate, value = _run(tiny_mx, inp)
    _check_all(tiny_mx, inp, out, gate, value)


@pytest.mark.parametrize("T", [300, 600])
def test_tiny_mxfp8_max_tokens_with_odd_token_tiles(T):
    """As the bf16 case: T = max_tokens with an odd number of 128-token
    tiles, so the last CTA pair's second tile (codes and scale atoms) lies
    in the staging buffers' padding."""
    case = Case(W.TINY_MXFP8, max_tokens=T)
    inp = case.step_inputs(T=T, step=T + 13)
    out, gate, value = _run(case, inp)
    _check_all(case, inp, out, gate, value)
    case.layer.close()


def test_tiny_mxfp8_lookup_then_forward(tiny_mx):
    inp = tiny_mx.step_inputs(T=48, step=5)
    out, _, _ = _run(tiny_mx, inp)
    tiny_mx.layer.lookup(inp["hash_ids"])
    out2 = tiny_mx.layer.forward(inp["hidden"], None, inp["token_mask"])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_mxfp8_decode_config(mx):
    inp = mx.step_inputs()
    out, gate, value = _run(mx, inp)
    _check_all(mx, inp, out, gate, value)


@pytest.mark.parametrize("T", [1, 100, 129])
def test_mxfp8_decode_shapes_ragged_T(mx, T):
    inp = mx.step_inputs(T=T, step=T)
    out, gate, value = _run(mx, inp)
    _check_all(mx, inp, out, gate, value)


def test_mxfp8_prefill_config_every_token(mx):
    """MXFP8 prefill (T = 4096, dim 7168) at every token: codes and scales
    bit for bit, the output against both oracle modes."""
    wl = W.MXFP8_PREFILL
    mx.wl = wl
    try:
        inp = mx.step_inputs()
        out, gate, value = _run(mx, inp)
        codes, scales = mx.layer.staged_mx(wl.T)
        torch.cuda.synchronize()
        ref_q = oracle_all(mx, inp, quantize_act=True)
        q_ref, s_ref = oracle.mx_quantize(ref_q["rows"].reshape(wl.T, -1))
        assert np.array_equal(codes.cpu().numpy(), q_ref)
        assert np.array_equal(scales.cpu().numpy(), s_ref)
        compare(mx, inp, out, ref_q, gate=gate, value=value, value_rtol=2.0 ** -8 + 1e-3,
                gate_rtol=1e-3)
        ref = oracle_all(mx, inp)
        compare(mx, inp, out, ref, gate=gate, value=value, value_rtol=5e-2, gate_rtol=5e-2,
                rounding=False)
        assert mx.layer.device_error() == 0
    finally:
        mx.wl = W.MXFP8_DECODE
