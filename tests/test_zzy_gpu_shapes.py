"""GPU parity on configurations the ABI admits beyond the named workloads:
hc_mult 1 with head_dim 128 (the fused grid shrinks to 128 CTAs of one
16-column granule each, some holding only value or only key columns), and
hc_mult 3 with 12 hash columns (K = 768; key runs that straddle two hc
copies).  Each at one token, a ragged decode size and a prefill size (three
128-token tiles, so the GEMM's last CTA pair reads padding) against the
oracle on every output, with the gate and value bars.  Runs after the
single-layer parity files (file order)."""
import pytest
import torch

import workloads as W
from engram_case import Case, compare

pytestmark = pytest.mark.gpu

ROWS12 = (1009, 1013, 1019, 1021, 1031, 1033, 1039, 1049, 1051, 1061, 1063, 1069)
SHAPES = {
    "h1_e128": W.Workload("h1_e128", T=16, dim=1024, hc_mult=1, max_ngram_size=3, n_heads=4,
                          head_dim=128, rows=W.TINY_ROWS, mask_p=0.75, tol=3e-2, seed=1321),
    "h3_c12": W.Workload("h3_c12", T=16, dim=2048, hc_mult=3, max_ngram_size=3, n_heads=6,
                         head_dim=64, rows=ROWS12, mask_p=0.75, tol=3e-2, seed=1322),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.fixture(scope="module", params=sorted(SHAPES))
def case(request):
    c = Case(SHAPES[request.param], max_tokens=512)
    yield c
    c.layer.close()


@pytest.mark.parametrize("T", [1, 37, 300])
def test_shape_matches_oracle(case, T):
    inp = case.step_inputs(T=T, step=T)
    out = case.layer.forward(inp["hidden"], inp["hash_ids"], inp["token_mask"])
    torch.cuda.synchronize()
    gate, value = case.layer.intermediates(T)
    torch.cuda.synchronize()
    ref = case.oracle(inp)
    # the prefill tiles store the value in bf16
    value_rtol = 1e-2 if T <= 256 else 2.0 ** -8 + 1e-3
    compare(case, inp, out, ref, gate=gate, value=value, value_rtol=value_rtol)
    assert case.layer.device_error() == 0
