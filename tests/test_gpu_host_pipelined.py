"""engram_forward_host_pipelined: host-buffer forwards whose input copies
overlap the previous call (and, with ENGRAM_HOST_DEFER_OUTPUT, whose output
copies overlap the next one).  Several calls in a row with different inputs
(the two device slots alternate) must give, bit for bit, what
engram_forward_host gives for the same inputs; so must calls captured into
a CUDA graph, where the entry point keeps every step on the caller's
stream."""
import pytest
import torch

import workloads as W
from engram_case import Case
from hashed_gram_engram_gb300 import EngramError, _lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _host_inputs(case, n, T):
    out = []
    for i in range(n):
        inp = case.step_inputs(T=T, step=40 + i)
        mask = inp["token_mask"]
        out.append((inp["hidden"].cpu().pin_memory(), inp["hash_ids"].cpu().pin_memory(),
                    None if mask is None else mask.cpu().pin_memory()))
    return out


def _serial(case, inputs):
    res = []
    for hid, ids, mask in inputs:
        o = torch.empty_like(hid).pin_memory()
        case.layer.forward_host(hid, ids, mask, o)
        torch.cuda.synchronize()
        res.append(o.clone())
    return res


@pytest.mark.parametrize("name, T", [("decode", 64), ("tiny", 16), ("tiny", 300)])
def test_back_to_back_calls_match_serial(name, T):
    wl = W.DECODE if name == "decode" else W.TINY
    case = Case(wl, max_tokens=T)
    inputs = _host_inputs(case, 5, T)
    ref = _serial(case, inputs)
    stream = torch.cuda.Stream()
    outs = [torch.empty_like(h).pin_memory() for h, _, _ in inputs]
    for (hid, ids, mask), o in zip(inputs, outs):  # no synchronisation in between
        case.layer.forward_host_pipelined(hid, ids, mask, o, stream=stream)
    stream.synchronize()
    for i, (o, r) in enumerate(zip(outs, ref)):
        assert torch.equal(o, r), f"call {i} differs from engram_forward_host"
    # one output buffer for every call: the last call's result remains
    shared = torch.empty_like(outs[0]).pin_memory()
    for hid, ids, mask in inputs:
        case.layer.forward_host_pipelined(hid, ids, mask, shared, stream=stream)
    stream.synchronize()
    assert torch.equal(shared, ref[-1])
    assert case.layer.device_error() == 0
    case.layer.close()


def test_graph_capture_keeps_the_calls_on_the_stream():
    case = Case(W.TINY, max_tokens=64)
    inputs = _host_inputs(case, 2, 64)
    ref = _serial(case, inputs)
    outs = [torch.empty_like(h).pin_memory() for h, _, _ in inputs]
    stream = torch.cuda.Stream()
    for (hid, ids, mask), o in zip(inputs, outs):  # (warm-up outside the capture)
        case.layer.forward_host_pipelined(hid, ids, mask, o, stream=stream)
    stream.synchronize()
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for (hid, ids, mask), o in zip(inputs, outs):
            case.layer.forward_host_pipelined(hid, ids, mask, o, stream=stream)
    g.replay()
    torch.cuda.synchronize()
    for o, r in zip(outs, ref):
        assert torch.equal(o, r)
    case.layer.close()


@pytest.mark.parametrize("name, T", [("decode", 64), ("tiny", 300)])
def test_deferred_output_lags_one_call_then_flushes(name, T):
    wl = W.DECODE if name == "decode" else W.TINY
    case = Case(wl, max_tokens=T)
    inputs = _host_inputs(case, 5, T)
    ref = _serial(case, inputs)
    stream = torch.cuda.Stream()
    outs = [torch.zeros_like(h).pin_memory() for h, _, _ in inputs]
    for i, ((hid, ids, mask), o) in enumerate(zip(inputs, outs)):
        case.layer.forward_host_pipelined(hid, ids, mask, o, stream=stream, defer_output=True)
        if i >= 1:  # the previous call's output is written once the stream gets here
            stream.synchronize()
            assert torch.equal(outs[i - 1], ref[i - 1]), f"call {i - 1}"
    case.layer.flush_host(stream)
    stream.synchronize()
    assert torch.equal(outs[-1], ref[-1])
    # back to ordered calls on the same slots
    last = torch.empty_like(outs[0]).pin_memory()
    hid, ids, mask = inputs[2]
    case.layer.forward_host_pipelined(hid, ids, mask, last, stream=stream)
    stream.synchronize()
    assert torch.equal(last, ref[2])
    with pytest.raises(EngramError) as e:
        _lib.engram_forward_host_pipelined(case.layer.handle, hid, ids, mask, last, T, 2, stream)
    assert e.value.code == _lib.ENGRAM_ERR_INVALID_ARG
    case.layer.close()
