"""GPU parity with an fp8 hash table: rows stored as e4m3 codes with one ue8m0
scale per 32 elements (class ParallelEngramEmbedding's storage), dequantized
to bf16 by the gather.

Bars: the staged (dequantized) rows equal the oracle's gather_e4m3 bit for
bit; the forward matches the oracle run on the same table at the
configuration's tolerance and at rounding level, gate and value within the
parity bar.  Covered: the fused decode kernel (T <= 128), the prefill tiles
(T > 256), MXFP8 wkv on top of an fp8 table, out-of-range ids, and the
decode-shaped table (1.07 GB of rows -> 0.54 GB of codes)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from engram_case import Case, compare
from hashed_gram_engram_gb300 import ENGRAM_DEVERR_BAD_HASH_ID

pytestmark = pytest.mark.gpu

TINY_MX_E4M3 = dataclasses.replace(W.TINY_MXFP8, name="tiny_mxfp8_e4m3_table",
                                   table_format="e4m3", seed=1244)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.fixture(scope="module")
def tiny():
    return Case(W.TINY_E4M3, max_tokens=1024)


@pytest.fixture(scope="module")
def decode():
    return Case(W.DECODE_E4M3, max_tokens=256)


def _run(case, inp):
    out = case.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    gate, value = case.layer.intermediates(inp["hidden"].shape[0])
    torch.cuda.synchronize()
    return out, gate, value


def _rows_exact(case, inp, ref, tokens=None):
    T = inp["hidden"].shape[0]
    rows = W.bits(case.layer.staged_rows(T)).reshape(T, -1)
    sel = slice(None) if tokens is None else tokens
    assert np.array_equal(rows[sel], ref["rows"].reshape(ref["rows"].shape[0], -1))


def test_table_storage_is_fp8(tiny):
    assert tiny.table.dtype == torch.uint8 and tiny.table_scale.dtype == torch.uint8
    assert tiny.table_scale.shape == (W.TINY_E4M3.total_rows, W.TINY_E4M3.head_dim // 32)


@pytest.mark.parametrize("T", [1, 16, 17, 100, 128])
def test_tiny_fused_path(tiny, T):
    inp = tiny.step_inputs(T=T, step=T)
    out, gate, value = _run(tiny, inp)
    ref = tiny.oracle(inp)
    _rows_exact(tiny, inp, ref)
    compare(tiny, inp, out, ref, gate=gate, value=value)
    assert tiny.layer.device_error() == 0


@pytest.mark.parametrize("T", [300, 1024])
def test_tiny_prefill_path(tiny, T):
    inp = tiny.step_inputs(T=T, step=T)
    out, gate, value = _run(tiny, inp)
    ref = tiny.oracle(inp)
    _rows_exact(tiny, inp, ref)
    # the prefill tiles store the value in bf16 (up to 2^-8 relative)
    compare(tiny, inp, out, ref, gate=gate, value=value, value_rtol=2.0 ** -8 + 1e-3)
    assert tiny.layer.device_error() == 0


@pytest.mark.parametrize("T", [16, 300])
def test_tiny_mxfp8_wkv_on_fp8_table(T):
    case = Case(TINY_MX_E4M3, max_tokens=512)
    inp = case.step_inputs(T=T, step=T)
    out, gate, value = _run(case, inp)
    ref_q = case.oracle(inp, quantize_act=True)
    value_rtol = 1e-3 if T <= 128 else 2.0 ** -8 + 1e-3
    compare(case, inp, out, ref_q, gate=gate, value=value, value_rtol=value_rtol,
            gate_rtol=1e-3)
    # the MXFP8 activations are the oracle's quantisation of the dequantized rows
    codes, scales = case.layer.staged_mx(T)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.mx_quantize(ref_q["rows"].reshape(T, -1))
    assert np.array_equal(codes.cpu().numpy(), q_ref)
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert case.layer.device_error() == 0
    case.layer.close()


def test_tiny_lookup_then_forward(tiny):
    T = 40
    inp = tiny.step_inputs(T=T, step=77)
    ref = tiny.oracle(inp)
    tiny.layer.lookup(inp["hash_ids"])
    out = tiny.layer.forward(inp["hidden"], None, inp["token_mask"])
    torch.cuda.synchronize()
    _rows_exact(tiny, inp, ref)
    compare(tiny, inp, out, ref)


def test_decode_config_full(decode):
    inp = decode.step_inputs()
    out, gate, value = _run(decode, inp)
    ref = decode.oracle(inp)
    _rows_exact(decode, inp, ref)
    res = compare(decode, inp, out, ref, gate=gate, value=value)
    assert decode.layer.device_error() == 0
    print("decode e4m3 table", res)
    # the lookup kernel's rows feed the same forward bit for bit
    decode.layer.lookup(inp["hash_ids"])
    out2 = decode.layer.forward(inp["hidden"], None, inp["token_mask"])
    torch.cuda.synchronize()
    _rows_exact(decode, inp, ref)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_decode_out_of_range_ids(decode):
    T = 32
    inp = decode.step_inputs(T=T, step=99)
    ids = inp["hash_ids"].clone()
    ids[3, 2] = W.DECODE_E4M3.rows[2]
    ids[9, 15] = -7
    inp["hash_ids"] = ids
    out, gate, value = _run(decode, inp)
    ref = decode.oracle(inp)
    assert ref["n_bad"] == 2
    _rows_exact(decode, inp, ref)
    compare(decode, inp, out, ref, gate=gate, value=value)
    assert decode.layer.device_error() & ENGRAM_DEVERR_BAD_HASH_ID


def test_decode_prefill_shape_sampled(decode):
    T = 256 + 44  # prefill tiles (T > 256 is beyond the fused kernel)
    case = Case(W.DECODE_E4M3, max_tokens=T)
    inp = case.step_inputs(T=T, step=5)
    out, gate, value = _run(case, inp)
    tokens = np.unique(np.r_[0, 1, 127, 128, 255, 256, T - 1,
                             np.random.default_rng(3).choice(T, 12)])
    ref = case.oracle(inp, tokens=tokens)
    _rows_exact(case, inp, ref, tokens=tokens)
    compare(case, inp, out, ref, tokens=tokens, gate=gate, value=value,
            value_rtol=2.0 ** -8 + 1e-3)
    case.layer.close()
