"""The fused decode kernel's launch plan, checked on the CPU for every shape
the ABI admits: the host code that engram_forward runs (read through
engram_debug_fused_plan, which touches no device) must keep every
shared-memory region inside the CTA's allocation, every MMA operand read
inside the token ring, the swizzled stages aligned, and the TMEM columns
within the 512 a CTA allocates.  These are the conditions whose violation
faults a GPU, so they are proven here rather than found there."""
import itertools

import pytest

from hashed_gram_engram_gb300 import _lib

TILE_ROWS_BYTES = 128 * 128  # one 128-token tile of a 128-byte k-block


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _cfg(dim, hc, ngram, heads, head_dim, mx):
    return _lib.engram_config(dim=dim, hc_mult=hc, max_ngram_size=ngram, n_heads=heads,
                              head_dim=head_dim, eps=1e-6, clamp=1e-6, max_tokens=256,
                              wkv_format=_lib.ENGRAM_WKV_MXFP8 if mx else _lib.ENGRAM_WKV_BF16,
                              table_location=_lib.ENGRAM_TABLE_DEVICE, device=0, table_format=0)


SHAPES = [  # dim, hc_mult, max_ngram_size, n_heads, head_dim
    (256, 2, 3, 4, 32), (512, 4, 3, 8, 64), (1024, 3, 3, 8, 64), (2048, 1, 3, 4, 32),
    (4096, 4, 3, 8, 64), (4096, 4, 4, 8, 64), (7168, 4, 3, 8, 64), (8192, 1, 3, 8, 64),
    (8192, 4, 3, 8, 64), (4096, 2, 3, 16, 128), (1024, 4, 3, 8, 16),
]
TOKENS = [1, 2, 15, 16, 17, 33, 63, 64, 65, 100, 127, 128, 129, 200, 255, 256]
SMS = [1, 7, 64, 132, 148, 152, 160]


def _check(p, T, mx, K):
    budget = p["smem_bytes"] - 1024  # after aligning the base to 1024 bytes
    assert 2 <= p["w_stages"] <= 12 and 4 <= p["x_stages"] <= 12
    assert p["mtiles"] == (T + 127) // 128 and p["Tn"] == (T + 15) // 16 * 16
    assert p["max_width"] <= 256 and p["max_width"] % 16 == 0
    # swizzled operands start on 1024-byte boundaries
    for k in ("w_stage_bytes", "x_stage_bytes", "x_off"):
        assert p[k] % 1024 == 0, k
    assert p["w_stage_bytes"] >= p["max_width"] * 128
    assert p["x_off"] == p["w_stages"] * p["w_stage_bytes"]
    # a token stage holds its copy; the MMA reads 16 KB per 128-token tile
    # from every stage base, the last stage's read inside the ring
    x_bytes = p["Tn"] * 128 if p["mtiles"] == 1 else 2 * TILE_ROWS_BYTES
    assert x_bytes <= p["x_stage_bytes"]
    assert p["x_stages"] * p["x_stage_bytes"] <= p["x_ring"]
    assert (p["x_stages"] - 1) * p["x_stage_bytes"] + TILE_ROWS_BYTES * p["mtiles"] <= p["x_ring"]
    assert p["x_off"] + p["x_ring"] <= p["qk_off"]
    assert p["qk_off"] + 256 * 4 <= p["bar_off"] and p["bar_off"] + 1024 <= budget
    # TMEM: accumulators at 0 (and 256 for a second tile or issuer); MXFP8
    # scale cells 16 columns per 128-byte k-block after the 256 accumulator ones
    if p["dual"]:
        assert p["mtiles"] == 1 and not mx
    if mx:
        assert T <= 128 and 256 + 16 * (K // 128) <= 512
    else:
        assert T <= 256


@pytest.mark.parametrize("shape", SHAPES)
def test_plan_invariants(shape):
    dim, hc, ngram, heads, E = shape
    K = (ngram - 1) * heads * E
    used = 0
    for mx, T, sms in itertools.product((False, True), TOKENS, SMS):
        if mx and E % 32:
            continue
        p = _lib.engram_debug_fused_plan(_cfg(dim, hc, ngram, heads, E, mx), T, sms)
        if not p["used"]:
            continue
        used += 1
        _check(p, T, mx, K)
        assert p["grid"] == min(sms, dim * (hc + 1) // 16)
    if dim * (hc + 1) // 16 // 152 <= 16:  # slices of at most 256 columns on 152 SMs
        assert used > 0, "the fused kernel serves none of these launches"


def test_decode_configuration_plan():
    """The decode step on 152 SMs: the plan the measurements describe."""
    p = _lib.engram_debug_fused_plan(_cfg(4096, 4, 3, 8, 64, False), 64, 152)
    assert p["used"] == 1 and p["grid"] == 152 and p["max_width"] == 144
    assert (p["x_stages"], p["w_stages"], p["dual"], p["mtiles"], p["k_blocks"]) == (12, 6, 1, 1, 16)
    mx = _lib.engram_debug_fused_plan(_cfg(7168, 4, 3, 8, 64, True), 64, 152)
    assert mx["used"] == 1 and mx["dual"] == 0 and mx["k_blocks"] == 8
    # beyond the fused kernel: T > 256 (bf16) and T > 128 (MXFP8) take the prefill path
    assert _lib.engram_debug_fused_plan(_cfg(4096, 4, 3, 8, 64, False), 257, 152)["used"] == 0
    assert _lib.engram_debug_fused_plan(_cfg(7168, 4, 3, 8, 64, True), 129, 152)["used"] == 0


def test_bad_arguments_are_rejected():
    out = (_lib.ctypes.c_int64 * _lib.ENGRAM_FUSED_PLAN_FIELDS)()
    cfg = _cfg(4096, 4, 3, 8, 64, False)
    L = _lib.load()
    assert L.engram_debug_fused_plan(None, 64, 152, out, 16) == _lib.ENGRAM_ERR_INVALID_ARG
    assert L.engram_debug_fused_plan(_lib.ctypes.byref(cfg), 0, 152, out, 16) == \
        _lib.ENGRAM_ERR_INVALID_ARG
    assert L.engram_debug_fused_plan(_lib.ctypes.byref(cfg), 64, 152, out, 15) == \
        _lib.ENGRAM_ERR_INVALID_ARG
