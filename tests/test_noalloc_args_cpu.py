"""engram_gate_noalloc's argument checks, on a machine without a GPU: every
malformed call returns its documented code before any device call.  The
device addresses below are fake and never dereferenced (the function only
compares them), so the module refuses to run where a GPU is visible: a call
that passed validation there would launch on them."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="fake device addresses: host-only checks")

OK, INVALID, CUDA_ERR, SCRATCH = 0, -1, -7, -8
T, H, D = 8, 4, 1024
HID, OUT, KV, Q, K = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x40100000


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from hashed_gram_engram_gb300 import _lib
    return _lib.load()


def strides(t, h, d=1):
    return (ctypes.c_int64 * 3)(t, h, d)


def call(lib, **kw):
    a = dict(hidden=HID, hs=strides(H * D, D), kv=KV, kv_stride=(H + 1) * D, q=Q, k=K,
             mask=None, out=OUT, os=strides(H * D, D), T=T, H=H, D=D, eps=1e-6, clamp=1e-6)
    a.update(kw)
    return lib.engram_gate_noalloc(a["hidden"], a["hs"], a["kv"], a["kv_stride"], a["q"], a["k"],
                                   a["mask"], a["out"], a["os"], a["T"], a["H"], a["D"],
                                   a["eps"], a["clamp"], None)


def test_a_well_formed_call_reaches_the_device_query(lib):
    # no GPU here: the first device call fails and nothing launches
    assert call(lib) == CUDA_ERR
    assert call(lib, T=0) == CUDA_ERR


@pytest.mark.parametrize("kw", [
    dict(T=-1), dict(H=0), dict(H=5), dict(D=128), dict(D=300), dict(D=8192 + 256),
    dict(eps=-1.0), dict(eps=float("nan")), dict(clamp=-1e-6), dict(clamp=float("nan")),
    dict(hidden=None), dict(out=None), dict(kv=None), dict(q=None), dict(k=None),
    dict(hs=None), dict(os=None),
    dict(hidden=HID + 8), dict(out=OUT + 8), dict(kv=KV + 2), dict(q=Q + 4), dict(k=K + 2),
    dict(hs=strides(H * D, D, 2)), dict(os=strides(H * D, D, 0)),
    dict(hs=strides(H * D + 4, D)), dict(os=strides(H * D, D + 4)), dict(hs=strides(-H * D, D)),
    dict(kv_stride=(H + 1) * D - 8), dict(kv_stride=(H + 1) * D + 4),
], ids=lambda kw: ",".join(f"{k}={v if not isinstance(v, ctypes.Array) else list(v)}"
                           for k, v in kw.items()))
def test_malformed_calls_are_rejected(lib, kw):
    assert call(lib, **kw) == INVALID


def test_overlaps(lib):
    span = ((T - 1) * H * D + (H - 1) * D + D) * 2
    # out may be hidden itself, with the same strides (reaches the device query)
    assert call(lib, out=HID) == CUDA_ERR
    # any other overlap with hidden or with kv is rejected
    assert call(lib, out=HID + span - 16) == INVALID
    assert call(lib, out=HID, os=strides(H * D, D + 8)) == INVALID
    assert call(lib, out=KV + 16) == INVALID
    assert call(lib, out=KV - span + 16) == INVALID
    # adjacent ranges do not overlap
    assert call(lib, out=HID + span) == CUDA_ERR
    assert call(lib, out=KV - span) == CUDA_ERR


def test_scratch_limit(lib):
    # T * H * (D / 256) partial slots, at most 131072, else nothing launches
    assert call(lib, T=131072 // (H * D // 256) + 1) == SCRATCH
    assert call(lib, T=131072 // (H * D // 256)) == CUDA_ERR
    one = dict(H=1, D=256, hs=strides(256, 256), os=strides(256, 256), kv_stride=512)
    assert call(lib, T=131073, **one) == SCRATCH
    assert call(lib, T=131072, **one) == CUDA_ERR


def test_output_rows_must_be_disjoint(lib):
    # rows of out that overlap each other would be written by several threads
    assert call(lib, os=strides(H * D, 0)) == INVALID
    assert call(lib, os=strides(D, D)) == INVALID
    assert call(lib, os=strides(0, D)) == INVALID
    # in place on a hidden broadcast over the copies: rejected for the same reason
    assert call(lib, hs=strides(H * D, 0), out=HID, os=strides(H * D, 0)) == INVALID
    # copy-major rows (a transposed view) are disjoint
    assert call(lib, os=strides(D, T * D)) == CUDA_ERR
    # one token or one copy: only the other stride matters
    assert call(lib, T=1, os=strides(0, D)) == CUDA_ERR
    assert call(lib, H=1, os=strides(D, 0), hs=strides(D, 0), kv_stride=2 * D) == CUDA_ERR


def test_output_must_not_alias_q_k_or_mask(lib):
    assert call(lib, out=Q) == INVALID
    assert call(lib, out=K - 16) == INVALID
    assert call(lib, mask=OUT + 64) == INVALID
    span = ((T - 1) * H * D + (H - 1) * D + D) * 2
    assert call(lib, mask=OUT + span) == CUDA_ERR
