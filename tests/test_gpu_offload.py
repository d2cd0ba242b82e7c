"""GPU parity of the offload configuration: the 17.2 GB hashed table in
pinned host memory (134,219,512 rows of 64 bf16), read by the GPU across
the host link during the gather; T = 256 decode shapes.  Skipped when the
host cannot pin the table."""
import numpy as np
import pytest
import torch

import workloads as W
from engram_case import Case, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.fixture(scope="module")
def offload():
    wl = W.OFFLOAD
    need = wl.total_rows * wl.head_dim * 2
    avail = W.host_memory_bytes()
    if avail is not None and avail < need + (8 << 30):
        pytest.skip(f"needs {need >> 30} GiB of pinned host memory, {avail >> 30} GiB free")
    case = Case(wl)
    assert not case.table.is_cuda and case.table.is_pinned()
    yield case
    case.layer.close()


def test_offload_config_full(offload):
    inp = offload.step_inputs()
    out = offload.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    gate, value = offload.layer.intermediates(W.OFFLOAD.T)
    torch.cuda.synchronize()
    ref = offload.oracle(inp)
    compare(offload, inp, out, ref, gate=gate, value=value)
    # the rows fetched across the host link are bit-exact
    rows = offload.layer.staged_rows(W.OFFLOAD.T)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(rows), ref["rows"].reshape(W.OFFLOAD.T, -1))
    assert offload.layer.device_error() == 0


def test_offload_lookup_rows_from_the_table_ends(offload):
    """Ids at both ends of every column's bucket, through the standalone
    gather (engram_lookup) and the fused forward."""
    wl = W.OFFLOAD
    T = 8
    inp = offload.step_inputs(T=T, step=3)
    ids = inp["hash_ids"].clone()
    for c, p in enumerate(wl.rows):
        ids[0, c] = 0
        ids[1, c] = p - 1
    inp["hash_ids"] = ids
    offload.layer.lookup(ids)
    rows = offload.layer.staged_rows(T)
    out = offload.layer.forward(inp["hidden"], None, inp["token_mask"])
    torch.cuda.synchronize()
    ref = offload.oracle(inp)
    assert np.array_equal(W.bits(rows), ref["rows"].reshape(T, -1))
    compare(offload, inp, out, ref)
