"""GPU: several layers' lookups staged ahead on the prefetcher's side stream
(class EngramPrefetch's start / forward / join, Engram.prepare_embeddings).

Each prefetched forward must equal that layer's plain forward bit for bit (the
same kernels on the same rows).  One layer, with a host-offloaded table, is
also compared with the oracle.  Ordering is tested directly: the hash ids
are written on the caller's stream behind a spin of a few milliseconds, so
lookups that did not wait for the caller's stream would gather stale ids.
Also covered: join and the plain fallback, and a CUDA-graph capture of a
whole prefetched step.  The wkv mode (engram_wkv: the projection alone, in
bf16, ahead on the side stream; the layer then runs only the gate and
residual) is checked against the oracle's kv and outputs.  Runs after the
other GPU tests (file order)."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from engram_case import Case, compare
from hashed_gram_engram_gb300 import EngramError, EngramPrefetch

pytestmark = pytest.mark.gpu

WLS = [dataclasses.replace(W.TINY, name="tiny_pf0", seed=1301),
       dataclasses.replace(W.TINY, name="tiny_pf1_host", seed=1302, table_location="host"),
       dataclasses.replace(W.TINY, name="tiny_pf2", seed=1303)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.fixture(scope="module")
def cases():
    cs = [Case(wl, max_tokens=512) for wl in WLS]
    yield cs
    for c in cs:
        c.layer.close()


def _inputs(cases, T, step):
    return [c.step_inputs(T=T, step=step) for c in cases]


def _plain(cases, inps):
    outs = [c.layer.forward(i["hidden"], i["hash_ids"], i["token_mask"])
            for c, i in zip(cases, inps)]
    torch.cuda.synchronize()
    return outs


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("T", [16, 300])  # fused decode kernel / prefill kernels
def test_prefetched_forwards_match_plain(cases, T):
    inps = _inputs(cases, T, step=T)
    ref = _plain(cases, inps)
    pf = EngramPrefetch([c.layer for c in cases])
    try:
        pf.start([i["hash_ids"] for i in inps])
        assert all(pf.pending(l) for l in range(3))
        outs = {}
        for l in (2, 0, 1):  # any order
            outs[l] = pf.forward(l, inps[l]["hidden"], None, inps[l]["token_mask"])
            assert not pf.pending(l)
        torch.cuda.synchronize()
        for l in range(3):
            assert _same(outs[l], ref[l]), l
        value_rtol = 1e-2 if T <= 256 else 2.0 ** -8 + 1e-3
        compare(cases[1], inps[1], outs[1], cases[1].oracle(inps[1]), value_rtol=value_rtol)
        for c in cases:
            assert c.layer.device_error() == 0
    finally:
        pf.close()


def test_start_orders_after_the_callers_stream(cases):
    T = 16
    inps = _inputs(cases, T, step=5)
    ref = _plain(cases, inps)
    ids = [torch.zeros_like(i["hash_ids"]) for i in inps]
    pf = EngramPrefetch([c.layer for c in cases])
    try:
        s = torch.cuda.current_stream()
        torch.cuda._sleep(20_000_000)  # a bounded spin (cycles) on s
        for d, i in zip(ids, inps):
            d.copy_(i["hash_ids"])
        pf.start(ids, stream=s)
        outs = [pf.forward(l, inps[l]["hidden"], None, inps[l]["token_mask"], stream=s)
                for l in range(3)]
        torch.cuda.synchronize()
        for l in range(3):
            assert _same(outs[l], ref[l]), l
    finally:
        pf.close()


def test_join_and_the_plain_fallback(cases):
    T = 40
    inps = _inputs(cases, T, step=9)
    ref = _plain(cases, inps)
    pf = EngramPrefetch([c.layer for c in cases])
    try:
        pf.start([i["hash_ids"] for i in inps])
        o0 = pf.forward(0, inps[0]["hidden"], None, inps[0]["token_mask"])
        with pytest.raises(EngramError):  # the staged T differs
            pf.forward(1, inps[1]["hidden"][:8], None, None)
        pf.join()
        assert not any(pf.pending(l) for l in range(3))
        with pytest.raises(EngramError):  # nothing staged any more: ids needed
            pf.forward(1, inps[1]["hidden"], None, inps[1]["token_mask"])
        o1 = pf.forward(1, inps[1]["hidden"], inps[1]["hash_ids"], inps[1]["token_mask"])
        o2 = pf.forward(2, inps[2]["hidden"], inps[2]["hash_ids"], inps[2]["token_mask"])
        torch.cuda.synchronize()
        for o, r in zip((o0, o1, o2), ref):
            assert _same(o, r)
    finally:
        pf.close()


def test_graph_capture_of_a_prefetched_step(cases):
    T = 16
    inps = _inputs(cases, T, step=13)
    ref = _plain(cases, inps)
    pf = EngramPrefetch([c.layer for c in cases])
    try:
        s = torch.cuda.Stream()
        outs = [torch.empty_like(i["hidden"]) for i in inps]
        ids = [i["hash_ids"] for i in inps]

        def step():
            pf.start(ids, stream=s)
            for l in (1, 2):
                pf.forward(l, inps[l]["hidden"], None, inps[l]["token_mask"], out=outs[l],
                           stream=s)
            pf.join(stream=s)  # layer 0 is joined, then run plainly
            pf.forward(0, inps[0]["hidden"], ids[0], inps[0]["token_mask"], out=outs[0],
                       stream=s)

        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for _ in range(3):
            for o in outs:
                o.zero_()
            g.replay()
            torch.cuda.synchronize()
            for l in range(3):
                assert _same(outs[l], ref[l]), l
    finally:
        pf.close()


# ---------------------------------------------------------------- wkv mode

def _kv_close(kv_gpu, kv_ref):
    """bf16 kv against the oracle's fp64 kv: the kernel rounds an fp32 sum,
    so at most one bf16 rounding (2^-8 relative) plus fp32 summation error."""
    got = kv_gpu.float().cpu().numpy().astype(np.float64)
    scale = np.abs(kv_ref).max()
    assert np.all(np.abs(got - kv_ref) <= 2.0 ** -8 * np.abs(kv_ref) + 1e-5 * scale)


@pytest.mark.parametrize("T", [1, 16, 100])
def test_wkv_matches_the_oracle_kv(cases, T):
    c = cases[0]
    inp = c.step_inputs(T=T, step=31 + T)
    kv = c.layer.wkv(inp["hash_ids"])
    torch.cuda.synchronize()
    _kv_close(kv, c.oracle(inp)["kv"])
    # the rows it staged serve a later forward
    out = c.layer.forward(inp["hidden"], None, inp["token_mask"])
    ref = c.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    assert _same(out, ref)


def test_wkv_decode_configuration():
    c = Case(W.DECODE, max_tokens=64)
    try:
        inp = c.step_inputs()
        kv = c.layer.wkv(inp["hash_ids"])
        torch.cuda.synchronize()
        _kv_close(kv, c.oracle(inp)["kv"])
        assert c.layer.device_error() == 0
    finally:
        c.layer.close()


def test_wkv_mxfp8():
    wl = dataclasses.replace(W.TINY_MXFP8, name="tiny_mx_pf", seed=1311)
    c = Case(wl, max_tokens=128)
    try:
        inp = c.step_inputs(T=40, step=3)
        kv = c.layer.wkv(inp["hash_ids"])
        torch.cuda.synchronize()
        _kv_close(kv, c.oracle(inp, quantize_act=True)["kv"])
    finally:
        c.layer.close()


@pytest.mark.parametrize("T", [16, 300])  # wkv ahead / beyond the fused range: lookups only
def test_prefetch_wkv_mode(cases, T):
    inps = _inputs(cases, T, step=40 + T)
    ref = _plain(cases, inps)
    pf = EngramPrefetch([c.layer for c in cases], wkv=True)
    try:
        pf.start([i["hash_ids"] for i in inps])
        outs = [pf.forward(l, inps[l]["hidden"], None, inps[l]["token_mask"]) for l in (1, 2, 0)]
        outs = [outs[2], outs[0], outs[1]]
        torch.cuda.synchronize()
        for l, c in enumerate(cases):
            if T > 256:  # the plain path, bit for bit
                assert _same(outs[l], ref[l]), l
            # kv in bf16 before the gate: the value is rounded as in the
            # prefill tiles
            compare(c, inps[l], outs[l], c.oracle(inps[l]), value_rtol=2.0 ** -8 + 1e-3)
            assert c.layer.device_error() == 0
    finally:
        pf.close()


def test_graph_capture_of_the_wkv_mode(cases):
    T = 16
    inps = _inputs(cases, T, step=57)
    pf = EngramPrefetch([c.layer for c in cases], wkv=True)
    try:
        s = torch.cuda.Stream()
        outs = [torch.empty_like(i["hidden"]) for i in inps]
        ids = [i["hash_ids"] for i in inps]

        def step():
            pf.start(ids, stream=s)
            for l in range(3):
                pf.forward(l, inps[l]["hidden"], None, inps[l]["token_mask"], out=outs[l],
                           stream=s)

        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        s.synchronize()
        first = [o.clone() for o in outs]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for _ in range(3):
            for o in outs:
                o.zero_()
            g.replay()
            torch.cuda.synchronize()
            for l in range(3):
                assert _same(outs[l], first[l]), l
    finally:
        pf.close()
