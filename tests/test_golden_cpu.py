"""The oracle against the hand-derived worked example in tests/golden
(Engram.forward and _engram_gate_finish_kernel; derivation in the fixture).
Gathered rows, kv and the bf16 outputs must match bit for bit; dot and gate
to double rounding."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_bits(values):
    """bf16 bit patterns of values that bf16 holds exactly (the float32
    pattern's top half; the bottom half must be zero)."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    assert not np.any(u & 0xFFFF), "fixture value not exact in bf16"
    return (u >> 16).astype(np.uint16)


@pytest.fixture(scope="module")
def ex():
    with open(os.path.join(HERE, "golden", "worked_example_forward.json")) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def res(ex):
    c = ex["config"]
    E = c["head_dim"]
    return oracle.forward(_bf16_bits(ex["table"]), np.asarray(ex["row_offset"], np.int64),
                          np.asarray(ex["rows"], np.int64),
                          np.asarray(ex["hash_ids"], np.int32), E, _bf16_bits(ex["wkv"]),
                          _bf16_bits(ex["hidden"]), _bf16_bits(ex["q_weight"]),
                          _bf16_bits(ex["k_weight"]), np.asarray(ex["token_mask"], np.uint8),
                          eps=c["eps"], clamp=c["clamp"])


def test_fixture_is_consistent(ex):
    c = ex["config"]
    C = (c["max_ngram_size"] - 1) * c["n_heads"]
    assert len(ex["rows"]) == C and ex["row_offset"] == [0] + list(np.cumsum(ex["rows"])[:-1])
    assert np.asarray(ex["wkv"]).shape == (c["dim"] * (c["hc_mult"] + 1), C * c["head_dim"])
    assert np.asarray(ex["hidden"]).shape == (c["T"], c["hc_mult"], c["dim"])
    # q and k enter the dot only through their product, which is 1 here
    assert np.all(np.asarray(ex["q_weight"]) * np.asarray(ex["k_weight"]) == 1)
    assert ex["cite"] and ex["derivation"]


def test_rows_and_bad_id(ex, res):
    c = ex["config"]
    assert res["n_bad"] == ex["expected"]["n_bad"]
    rows = res["rows"].reshape(c["T"], -1)
    assert np.array_equal(rows, _bf16_bits(ex["expected"]["rows"]))


def test_kv(ex, res):
    assert np.array_equal(res["kv"], np.asarray(ex["expected"]["kv"], np.float64))


def test_dot_and_gate(ex, res):
    dot = np.asarray(ex["expected"]["dot"], np.float64)
    gate = np.asarray(ex["expected"]["gate"], np.float64)
    assert np.allclose(res["dot"], dot, rtol=0, atol=4e-16 * 4)
    assert np.allclose(res["gate"], gate, rtol=0, atol=4e-16)
    # dot = 0 takes the positive branch: sigmoid(+0.001), not sigmoid(0)
    assert res["gate"][2, 0] > 0.5


def test_out_bits(ex, res):
    exp = _bf16_bits(ex["expected"]["out"])
    assert np.array_equal(res["out_bf16"], exp)
    # the masked token keeps hidden's -0.0
    assert res["out_bf16"][3, 1, 0] == 0x8000


def test_fixture_regenerates_from_its_derivation(ex):
    """The expected block is what tests/golden/derive_worked_example.py
    computes from the fixture's inputs in exact arithmetic (fractions and
    50-digit decimals, no oracle code)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "derive_worked_example", os.path.join(HERE, "golden", "derive_worked_example.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.derive(ex) == ex["expected"]
