"""Host-side checks of the C ABI (no GPU needed): the library builds, loads
and exports every entry point include/engram.h declares, the host-only
layout function agrees with the oracle, and the product package has no
route to the oracle."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*int\s+(engram_\w+)\s*\(", src, re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from hashed_gram_engram_gb300 import _lib
    return _lib.load()


def test_library_exports_every_declared_symbol(lib):
    from hashed_gram_engram_gb300 import _lib
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert declared == set(_lib.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(engram_\w+)$", out, re.M))
    assert declared <= exported


def test_library_targets_sm103a_only(lib):
    from hashed_gram_engram_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def test_layout_entry_point_matches_oracle(lib):
    for vocab, ng, heads, layers in ((2 ** 19, 3, 8, 1), (1000, 4, 3, 3), (2 ** 23, 3, 8, 1)):
        from hashed_gram_engram_gb300 import engram_layout
        p, o = engram_layout(vocab, ng, heads, layers)
        rp, ro = oracle.layout(vocab, ng, heads, layers)
        assert np.array_equal(np.array(p), rp) and np.array_equal(np.array(o), ro)
    assert list(engram_layout(2 ** 19, 3, 8)[0][0]) == list(W.PRIMES_2POW19)


def test_layout_rejects_bad_arguments(lib):
    buf = (ctypes.c_int64 * 8)()
    assert lib.engram_layout(0, 3, 4, 1, buf, buf) == -1
    assert lib.engram_layout(100, 1, 4, 1, buf, buf) == -1
    assert lib.engram_layout(100, 3, 4, 1, None, buf) == -1


def test_null_handle_arguments_are_rejected_without_a_gpu(lib):
    st = (ctypes.c_int64 * 3)(0, 0, 1)
    assert lib.engram_lookup(None, None, 0, 1, 0, None) == -1
    assert lib.engram_forward(None, None, st, None, 0, None, None, st, 1, None) == -1
    assert lib.engram_destroy(None) == 0
    out = ctypes.c_void_p()
    assert lib.engram_create(None, None, ctypes.byref(out)) == -1
    assert out.value is None
    assert lib.engram_forward_host(None, None, None, None, None, 1, None) == -1
    assert lib.engram_forward_host_pipelined(None, None, None, None, None, 1, 0, None) == -1
    assert lib.engram_forward_host_flush(None, None) == -1


def test_prefetch_arguments_are_rejected_without_a_gpu(lib):
    out = ctypes.c_void_p()
    none = (ctypes.c_void_p * 2)(None, None)
    assert lib.engram_prefetch_create(None, 1, 0, ctypes.byref(out)) == -1
    assert lib.engram_prefetch_create(none, 0, 0, ctypes.byref(out)) == -1
    assert lib.engram_prefetch_create(none, 2, 2, ctypes.byref(out)) == -1  # unknown flag
    assert lib.engram_prefetch_create(none, 2, 0, ctypes.byref(out)) == -1  # null handles
    assert lib.engram_prefetch_create(none, 2, 0, None) == -1
    assert lib.engram_wkv(None, None, 0, None, 0, 1, None) == -1
    assert out.value is None
    st = (ctypes.c_int64 * 3)(0, 0, 1)
    assert lib.engram_prefetch_start(None, none, st, 1, 1, None) == -1
    assert lib.engram_prefetch_forward(None, 0, None, st, None, 0, None, None, st, 1,
                                       None) == -1
    assert lib.engram_prefetch_join(None, None) == -1
    assert lib.engram_prefetch_pending(None, 0) == -1
    assert lib.engram_prefetch_destroy(None) == 0
    assert lib.engram_debug_barrier_skew(None, 1) == -1


def test_product_package_never_reaches_the_oracle():
    pkg = os.path.join(ROOT, "hashed_gram_engram_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in src, f"{fn} mentions the oracle"


def _header():
    return open(os.path.join(ROOT, "include", "engram.h")).read()


def test_binding_constants_match_the_header():
    from hashed_gram_engram_gb300 import _lib
    defines = dict(re.findall(r"^#define\s+(ENGRAM_\w+)\s+\(?(-?\d+)u?\)?", _header(), re.M))
    assert defines, "no #define constants found"
    for name, value in defines.items():
        assert hasattr(_lib, name), f"{name} missing from the binding"
        assert getattr(_lib, name) == int(value), name


def test_binding_structs_match_the_header_layout(tmp_path):
    """Field order, offsets and sizes of the two ABI structs: the C compiler's
    view (a probe compiled against include/engram.h) against ctypes'."""
    from hashed_gram_engram_gb300 import _lib
    structs = {"engram_config": _lib.engram_config, "engram_weights": _lib.engram_weights}
    hdr = _header()
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "engram.h"', "int main(void) {"]
    for sname, cls in structs.items():
        body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (sname, sname), hdr, re.S).group(1)
        body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
        fields = re.findall(r"(\w+)\s*;", body)
        assert fields == [f for f, _ in cls._fields_], sname
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (sname, sname))
        for f in fields:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (sname, f, sname, f))
    lines.append("return 0; }")
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o",
                    str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for sname, cls in structs.items():
        assert int(got[sname]) == ctypes.sizeof(cls), sname
        for f, _ in cls._fields_:
            assert int(got[f"{sname}.{f}"]) == getattr(cls, f).offset, f"{sname}.{f}"


def test_create_validates_the_table_format_without_a_gpu(lib):
    """engram_create checks its arguments before touching a device: an fp8
    table needs its scales and a head_dim that is a multiple of 32, and
    table_format takes only the two defined values.  The device pointers are
    fake (aligned, never dereferenced); rows and row_offset are real host
    arrays."""
    from hashed_gram_engram_gb300 import _lib
    rows = np.array([1009, 1019, 1033, 1049, 1061, 1069, 1093, 1103] * 2, np.int64)  # >= C
    off = W.row_offsets(rows)
    fake = 1 << 40

    def create(table_format, head_dim, table_scale):
        n_heads = 8 * 32 // (2 * head_dim) if head_dim <= 128 else 1
        cfg = _lib.engram_config(dim=256, hc_mult=2, max_ngram_size=3, n_heads=n_heads,
                                 head_dim=head_dim, eps=1e-6, clamp=1e-6, max_tokens=16,
                                 wkv_format=_lib.ENGRAM_WKV_BF16,
                                 table_location=_lib.ENGRAM_TABLE_DEVICE, device=0,
                                 table_format=table_format)
        w = _lib.engram_weights(table=fake, row_offset=off.ctypes.data, rows=rows.ctypes.data,
                                wkv=fake, wkv_scale=None, q_weight=fake, k_weight=fake,
                                table_scale=table_scale)
        out = ctypes.c_void_p()
        rc = lib.engram_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(out))
        assert out.value is None
        return rc

    # 2 * n_heads hash columns of head_dim: K = 2 * n_heads * head_dim = 512
    assert create(_lib.ENGRAM_TABLE_FORMAT_E4M3, 32, None) == _lib.ENGRAM_ERR_INVALID_ARG
    assert create(2, 32, fake) == _lib.ENGRAM_ERR_INVALID_ARG
    assert create(-1, 32, None) == _lib.ENGRAM_ERR_INVALID_ARG
    assert create(_lib.ENGRAM_TABLE_FORMAT_E4M3, 16, fake) == _lib.ENGRAM_ERR_UNSUPPORTED
