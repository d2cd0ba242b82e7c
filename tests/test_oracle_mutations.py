"""The pins catch plausible slips: each case plants one mistake in a copy of
the oracle's C source, builds it into a temporary library, points the
oracle's wrappers at it, and checks that the pin written for that function
now fails.  The committed oracle is never modified."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import oracle.oracle as oracle_mod
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle_mod.__file__), "engram_oracle.c")

# (name, text in the C source, planted replacement, the pin that must fail)
MUTANTS = [
    ("qact: activation scale read with the weight's block index",
     "oracle_e8m0_to_f64(As[t * kb + k / 32]);",
     "oracle_e8m0_to_f64(As[(n / 32) * kb + k / 32]);",
     "test_wkv_mxfp8_qact_matches_numpy_matmul"),
    ("qact: activation scale dropped",
     "oracle_e4m3_to_f64(Aq[t * K + k]) *\n                           oracle_e8m0_to_f64(As[t * kb + k / 32]);",
     "oracle_e4m3_to_f64(Aq[t * K + k]);",
     "test_wkv_mxfp8_qact_matches_numpy_matmul"),
    ("qact: weight scale per k-block only",
     "double w = oracle_e4m3_to_f64(Wq[n * K + k]) *\n                           oracle_e8m0_to_f64(Ws[(n / 32) * kb + k / 32]);\n                acc += a * w;",
     "double w = oracle_e4m3_to_f64(Wq[n * K + k]) *\n                           oracle_e8m0_to_f64(Ws[k / 32]);\n                acc += a * w;",
     "test_wkv_mxfp8_qact_matches_numpy_matmul"),
    ("qact: transposed weight codes",
     "double w = oracle_e4m3_to_f64(Wq[n * K + k]) *\n                           oracle_e8m0_to_f64(Ws[(n / 32) * kb + k / 32]);\n                acc += a * w;",
     "double w = oracle_e4m3_to_f64(Wq[(k % N) * K + (n % K)]) *\n                           oracle_e8m0_to_f64(Ws[(n / 32) * kb + k / 32]);\n                acc += a * w;",
     "test_wkv_mxfp8_qact_matches_numpy_matmul"),
    ("mx_quantize: scale one power of two too large",
     "while (e < 127 && amax > 448.0 * ldexp(1.0, e)) ++e;",
     "while (e < 127 && amax > 448.0 * ldexp(1.0, e)) ++e;\n                ++e;",
     "test_mx_quantize_scale_is_minimal_and_codes_match_torch"),
    ("wkv_mxfp8: weight scale with the columns' block index swapped",
     "oracle_e8m0_to_f64(Ws[(n / 32) * kb + k / 32]);\n                acc += oracle_bf16_to_f64",
     "oracle_e8m0_to_f64(Ws[(k / 32) % (N / 32) * kb + (n / 32) % kb]);\n                acc += oracle_bf16_to_f64",
     "test_wkv_mxfp8_matches_numpy_matmul"),
]


@pytest.fixture
def mutant(tmp_path, monkeypatch):
    def make(old, new):
        src = open(SRC).read()
        assert src.count(old) == 1, old
        path = tmp_path / "engram_oracle.c"
        path.write_text(src.replace(old, new))
        monkeypatch.setattr(oracle_mod, "_SRC", str(path))
        monkeypatch.setattr(oracle_mod, "_OUT_DIR", str(tmp_path))
        monkeypatch.setattr(oracle_mod, "_SO", str(tmp_path / "liboracle.so"))
        monkeypatch.setattr(oracle_mod, "_lib", None)
    yield make
    # the next test loads the committed oracle again
    oracle_mod._lib = None


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,old,new,pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_slip_fails_its_pin(mutant, name, old, new, pin):
    mutant(old, new)
    with pytest.raises(AssertionError):
        getattr(pins, pin)()


def test_committed_oracle_passes_the_same_pins():
    for pin in sorted({m[3] for m in MUTANTS}):
        getattr(pins, pin)()
