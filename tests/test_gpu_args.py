"""engram_forward's argument checks that need a live handle (so a GPU): an
output whose rows overlap each other, or that overlaps the hash ids or the
token mask, is refused with ENGRAM_ERR_INVALID_ARG before anything is
launched, and the handle stays usable."""
import ctypes

import pytest
import torch

import workloads as W
from engram_case import Case
from hashed_gram_engram_gb300 import _lib

pytestmark = pytest.mark.gpu
INVALID = -1


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _call(c, hidden, hs, ids, ids_stride, mask, out, os, T):
    L = _lib.load()
    st = lambda s: (ctypes.c_int64 * 3)(*s)  # noqa: E731
    return L.engram_forward(c.layer.handle, ctypes.c_void_p(hidden.data_ptr()), st(hs),
                            ctypes.c_void_p(ids.data_ptr()), int(ids_stride),
                            None if mask is None else ctypes.c_void_p(mask.data_ptr()),
                            ctypes.c_void_p(out.data_ptr()), st(os), int(T), None)


def test_overlapping_outputs_are_refused():
    c = Case(W.TINY)
    try:
        inp = c.step_inputs()
        hid, ids, mask = inp["hidden"], inp["hash_ids"], inp["token_mask"]
        T, H, D = hid.shape
        out = torch.empty_like(hid)
        ok = (H * D, D, 1)
        assert _call(c, hid, ok, ids, ids.stride(0), mask, out, ok, T) == 0
        torch.cuda.synchronize()
        ref = out.clone()
        # rows of out overlapping each other
        assert _call(c, hid, ok, ids, ids.stride(0), mask, out, (H * D, 0, 1), T) == INVALID
        assert _call(c, hid, ok, ids, ids.stride(0), mask, out, (D, D, 1), T) == INVALID
        # out over the hash ids or the mask
        big = torch.empty(T * H * D + 4096, dtype=torch.bfloat16, device=hid.device)
        ids_in = big.view(torch.int32)[: T * ids.shape[1]].view(T, -1)
        ids_in.copy_(ids)
        assert _call(c, hid, ok, ids_in, ids_in.stride(0), mask, big, ok, T) == INVALID
        mask_in = big.view(torch.uint8)[1024:1024 + T]
        mask_in.copy_(mask)
        assert _call(c, hid, ok, ids, ids.stride(0), mask_in, big, ok, T) == INVALID
        # copy-major rows are accepted and give the same result
        outT = torch.empty((H, T, D), dtype=hid.dtype, device=hid.device)
        assert _call(c, hid, ok, ids, ids.stride(0), mask, outT, (D, T * D, 1), T) == 0
        torch.cuda.synchronize()
        assert torch.equal(outT.transpose(0, 1).view(torch.int16), ref.view(torch.int16))
        assert c.layer.device_error() == 0
    finally:
        c.layer.close()
