"""Failure detection on the GPU, without a fault: the fused decode kernel's
grid barriers are made to wait for arrivals that never come (a launch counter
skewed by engram_debug_barrier_skew).  Each bounded wait gives up after its
limit; the launch reports ENGRAM_DEVERR_TIMEOUT and returns; the host read of
the flag resets the counters; and the next launch matches a clean run bit for
bit, so the context stayed usable.  Nothing faults, traps or hangs."""
import time

import pytest
import torch

import workloads as W
from engram_case import Case
from hashed_gram_engram_gb300 import ENGRAM_DEVERR_TIMEOUT, _lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def test_barrier_wait_expiry_is_reported_and_recovered():
    c = Case(W.TINY, max_tokens=64)
    try:
        inp = c.step_inputs(T=16, step=3)
        ref = c.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
        torch.cuda.synchronize()
        assert c.layer.device_error() == 0
        _lib.engram_debug_barrier_skew(c.layer.handle, 5)
        t0 = time.perf_counter()
        c.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        bits = c.layer.device_error()  # reads, clears, resets the barrier counters
        assert bits & ENGRAM_DEVERR_TIMEOUT
        assert 0.5 < elapsed < 60  # one or two 1 s limits ran out
        out = c.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert c.layer.device_error() == 0
    finally:
        c.layer.close()
