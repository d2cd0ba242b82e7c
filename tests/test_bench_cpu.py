"""Host logic of the benchmark: the algorithmic bytes behind every roofline
fraction, derived here component by component from the workload shapes, and
the stored-traffic lookup that withholds an ncu figure once the kernel's
sources have changed."""
import bench
import workloads as W


def _bytes(T, D, H, C, E, N, K, mx=False, mask=False, offload=False):
    w = N * K * (1 if mx else 2) + ((N // 32) * (K // 32) if mx else 0)
    hidden = 2 * T * H * D * 2            # read and written, bf16
    rows = 0 if offload else T * C * E * 2  # the gathered rows, bf16
    ids = T * C * 4
    qk = 2 * H * D * 2
    return w + hidden + rows + ids + qk + (T if mask else 0)


def test_algorithmic_bytes_per_workload():
    # the decode step: wkv 41.9 MB, hidden in and out 4.19 MB, rows 131 KB
    assert bench.algorithmic_bytes(W.DECODE) == _bytes(64, 4096, 4, 16, 64, 20480, 1024) \
        == 46_338_048
    assert bench.algorithmic_bytes(W.PREFILL) == \
        _bytes(8192, 4096, 4, 16, 64, 20480, 1024, mask=True) == 596_189_184
    assert bench.algorithmic_bytes(W.MXFP8_DECODE) == \
        _bytes(64, 7168, 4, 16, 64, 35840, 1024, mx=True) == 44_325_888
    assert bench.algorithmic_bytes(W.MXFP8_PREFILL) == \
        _bytes(4096, 7168, 4, 16, 64, 35840, 1024, mx=True) == 515_263_488
    # offload: the rows cross the host link, not HBM
    assert bench.algorithmic_bytes(W.OFFLOAD) == \
        _bytes(256, 4096, 4, 16, 64, 20480, 1024, offload=True) == 58_802_176
    assert bench.row_bytes(W.OFFLOAD) == 256 * 16 * 64 * 2 == 524_288
    # an fp8 table's rows: one code byte per element plus a scale per 32
    assert bench.row_bytes(W.DECODE_E4M3) == 64 * 1024 + 64 * 1024 // 32


def test_gate_kernel_bytes_per_workload():
    # hidden read and output written (bf16), the bf16 value row, one 16-byte
    # partial record per token, copy and 256-column tile (MXFP8: two per
    # 224-column tile), the fp32 gate, and the mask byte
    T, H, D = 8192, 4, 4096
    assert bench.gate_ring_bytes(W.PREFILL, 256) == \
        2 * T * H * D * 2 + T * D * 2 + T * H * (D // 256) * 16 + T * H * 4 + T == 612_507_648
    T, D = 4096, 7168
    assert bench.gate_ring_bytes(W.MXFP8_PREFILL, 224) == \
        2 * T * H * D * 2 + T * D * 2 + T * H * 2 * (D // 224) * 16 + T * H * 4 == 545_325_056


def test_profile_names_follow_kernel_and_workload():
    assert bench.profile_path("wkv_gemm_kernel", W.PREFILL).endswith(
        "profiles/wkv_gemm_kernel_prefill_T8192.md")
    assert bench.profile_path("gate_ring_kernel", W.MXFP8_PREFILL).endswith(
        "profiles/gate_ring_kernel_mxfp8_prefill_T4096.md")


def test_source_digest_ignores_comments_only():
    d = bench.source_digest(bench.DECODE_SOURCES)
    assert len(d) == 12 and d == bench.source_digest(bench.DECODE_SOURCES)
    assert d != bench.source_digest(("gather.cu",))


def test_stored_traffic_needs_matching_sources(tmp_path):
    d = bench.source_digest(bench.DECODE_SOURCES)
    good = tmp_path / "good.md"
    good.write_text("# summary\n\ntraffic: kernel=k source_sha256=%s dram_bytes_per_launch=123\n" % d)
    assert bench.stored_traffic(str(good), bench.DECODE_SOURCES) == 123
    stale = tmp_path / "stale.md"
    stale.write_text("traffic: kernel=k source_sha256=000000000000 dram_bytes_per_launch=123\n")
    assert bench.stored_traffic(str(stale), bench.DECODE_SOURCES) is None
    assert bench.stored_traffic(str(tmp_path / "missing.md"), bench.DECODE_SOURCES) is None
    broken = tmp_path / "broken.md"
    broken.write_text("traffic: kernel=k source_sha256=%s\n" % d)
    assert bench.stored_traffic(str(broken), bench.DECODE_SOURCES) is None
