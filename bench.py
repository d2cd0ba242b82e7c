"""Benchmark of the Engram forward on GB300: one JSON line on rank 0.

A step is one whole forward (gather, wkv projection, gate and residual) of
one batch of synthetic inputs resident in HBM, through the C ABI.  The
headline workload is the decode step (T = 64, dim 4096, hc_mult 4, 16 hash
columns of head_dim 64, bf16 wkv [20480, 1024]); the prefill step
(T = 8192) is reported alongside.  Decode steps rotate over several
independently seeded layers whose weights together exceed the 129 MB L2,
so every step reads its weights from HBM; the rotation is captured in a
CUDA graph and timed with CUDA events on its stream.  The single-step
latency with L2 flushed (a 512 MB write) before every step is reported
too.  Alongside: the MXFP8 decode (T = 64, dim 7168) and prefill
(T = 4096) steps, the offload step (T = 256, the 17 GB table in
pinned host memory, every gathered row crossing the host link), and the
decode and offload steps again with an fp8 table (e4m3 rows with ue8m0
scales per 32 elements, dequantized by the gather: half the row bytes).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica on its own GPU (tokens are
independent: weak scaling, no collective in the data path); the value is
the tokens of all ranks over the slowest rank's time.  --impl reference
times the CPU oracle (rank 0 only) on a bounded sample of the same step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Engram forward tokens/s (decode step, T=64)"
L2_FLUSH_BYTES = 512 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-mxfp8", action="store_true", help="skip the MXFP8 decode and prefill")
    p.add_argument("--no-offload", action="store_true",
                   help="skip the offload workloads (17 GB / 8.9 GB pinned host tables)")
    p.add_argument("--no-e4m3-table", action="store_true",
                   help="skip the workloads whose hash table is fp8 (e4m3 + ue8m0 per 32)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--ref-seconds", type=float, default=90.0,
                   help="wall time the reference arm's warm-up and timed steps aim for")
    p.add_argument("--layers", type=int, default=6)
    p.add_argument("--min-ms", type=float, default=20.0,
                   help="least total replay time per timed workload (the median of at least "
                        "5 replays is reported); 0 for short profiler runs")
    p.add_argument("--case", choices=["decode", "prefill", "mxfp8_decode", "mxfp8_prefill"],
                   default=None,
                   help="only run W + K plain forwards of one layer of that workload (the "
                        "small case profilers capture) and print a one-line summary")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def cpu_oracle_tokens_per_s(wl, case_host, inputs_host, seconds, max_tokens=None):
    """The oracle as it stands on this host's cores (single-threaded C)."""
    import numpy as np
    import oracle
    T = inputs_host["hidden"].shape[0]
    n = T if max_tokens is None else min(T, max_tokens)
    done, t0 = 0, time.perf_counter()
    start = 0
    while True:
        idx = np.arange(start, start + n) % T
        start += n
        oracle.forward(case_host["table"], case_host["row_offset"], case_host["rows"],
                       np.ascontiguousarray(inputs_host["ids"][idx]), wl.head_dim,
                       case_host["wkv"], inputs_host["hidden"][idx], case_host["q"],
                       case_host["k"], None if inputs_host["mask"] is None
                       else inputs_host["mask"][idx], eps=wl.eps, clamp=wl.clamp)
        done += n
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el, done, el


def decode_config(wl):
    """The decode workload's keys, shared by both arms' JSON lines."""
    return {"workload": wl.name, "T": wl.T, "dim": wl.dim, "hc_mult": wl.hc_mult,
            "n_hash_cols": wl.n_hash_cols, "head_dim": wl.head_dim,
            "table_rows": wl.total_rows, "wkv": f"bf16 [{wl.N}, {wl.K}]", "mask": None}


def run_reference(args):
    """CPU oracle as the reference arm: bounded samples of the decode step."""
    import numpy as np
    import torch
    import workloads as W
    rank, _, world = dist_env()
    if rank != 0:
        return
    wl = W.DECODE
    # inputs on the host; the table only needs the rows the sample touches,
    # but the oracle indexes the full concatenated table as the layer does
    table = W.make_table(wl, "cpu")
    wts = W.make_weights(wl, "cpu")
    step = W.make_step_inputs(wl, "cpu")
    host = dict(table=W.bits(table), row_offset=W.row_offsets(wl.rows),
                rows=np.asarray(wl.rows, np.int64), wkv=W.bits(wts["wkv"]),
                q=W.bits(wts["q_weight"]), k=W.bits(wts["k_weight"]))
    inp = dict(hidden=W.bits(step["hidden"]), ids=step["hash_ids"].numpy(), mask=None)
    # size the per-step sample so that warmup + steps take about --ref-seconds
    per_tok, _, _ = cpu_oracle_tokens_per_s(wl, host, inp, 0.0, max_tokens=1)
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.T, budget * per_tok)))
    for _ in range(args.warmup):
        cpu_oracle_tokens_per_s(wl, host, inp, 0.0, max_tokens=n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_tokens_per_s(wl, host, inp, 0.0, max_tokens=n)
    el = time.perf_counter() - t0
    value = args.steps * n / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(decode_config(wl), tokens_per_step_sample=n,
                       seeds={"layers": [int(wl.seed)],
                              "generator": "torch.Generator.manual_seed per tensor kind"}),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} of the {wl.T} decode-step tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def source_digest(names):
    """sha256 (12 hex) of kernel sources with comments and whitespace removed,
    to tell whether a stored ncu figure still describes the code that runs
    (an edit of a comment does not change the kernel)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "hashed_gram_engram_gb300", "csrc", n)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                 # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:12]


DECODE_SOURCES = ("decode_fused.cu", "ptx.cuh", "internal.h")
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_fused_kernel_decode_T64.md")
GEMM_SOURCES = ("wkv_gemm.cu", "ptx.cuh", "internal.h")
GATE_SOURCES = ("gate.cu", "ptx.cuh", "internal.h")


def profile_path(kernel, wl):
    """The committed ncu summary of a kernel on a workload."""
    return os.path.join(ROOT, "profiles", f"{kernel}_{wl.name}_T{wl.T}.md")


def stored_traffic(path, sources):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    summary is missing or was taken on other kernel sources."""
    try:
        for line in open(path):
            if line.startswith("traffic:"):
                kv = dict(x.split("=", 1) for x in line.split()[1:])
                if kv.get("source_sha256") == source_digest(sources):
                    return int(kv["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def reduce_max(x, world, device):
    """The largest of every rank's x (the slowest rank's time sets the job's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_layer(W, Engram, wl, device_index, max_tokens, layer_seed, table=None):
    """One layer of workload wl with its own seed; a given table is shared
    (for an e4m3 table, the pair (codes, scales))."""
    import dataclasses
    wl_l = dataclasses.replace(wl, seed=wl.seed + 101 * layer_seed)
    if table is None:
        table = (W.make_table(wl_l, "cuda"), W.make_table_scale(wl_l, "cuda"))
    elif not isinstance(table, tuple):
        table = (table, None)
    table, table_scale = table
    wts = W.make_weights(wl_l, "cuda")
    wts["table_scale"] = table_scale
    layer = Engram(dim=wl.dim, hc_mult=wl.hc_mult, max_ngram_size=wl.max_ngram_size,
                   n_heads=wl.n_heads, head_dim=wl.head_dim, max_tokens=max_tokens,
                   table=table, rows=wl.rows, row_offset=W.row_offsets(wl.rows),
                   wkv=wts["wkv"], wkv_scale=wts["wkv_scale"], q_weight=wts["q_weight"],
                   k_weight=wts["k_weight"], eps=wl.eps, clamp=wl.clamp, device=device_index,
                   table_scale=table_scale)
    return wl_l, layer, table, wts


def algorithmic_bytes(wl):
    """HBM bytes one forward of wl must move: wkv (and its scales), hidden in
    and out, the gathered rows (from HBM unless the table is offloaded),
    ids, the token mask (one byte per token, when there is one), q and k."""
    mx = wl.wkv_format == "mxfp8"
    b = (wl.N * wl.K * (1 if mx else 2) + 2 * wl.T * wl.hc_mult * wl.dim * 2
         + wl.T * wl.n_hash_cols * 4 + 2 * wl.hc_mult * wl.dim * 2)
    if wl.mask_p is not None:
        b += wl.T
    if mx:
        b += (wl.N // 32) * (wl.K // 32)
    if wl.table_location != "host":
        b += row_bytes(wl)
    return b


def gate_ring_bytes(wl, tile_cols):
    """HBM bytes of the prefill gate kernel: hidden in, output out, the bf16
    value, the GEMM's gate-partial records (16 bytes per token, copy and
    record; MXFP8 writes two per tile), the fp32 gate it stores and the
    token mask."""
    records = (2 if wl.wkv_format == "mxfp8" else 1) * (wl.dim // tile_cols)
    b = (2 * wl.T * wl.hc_mult * wl.dim * 2 + wl.T * wl.dim * 2
         + wl.T * wl.hc_mult * records * 16 + wl.T * wl.hc_mult * 4)
    if wl.mask_p is not None:
        b += wl.T
    return b


def row_bytes(wl):
    """Bytes of the T x C gathered rows: bf16, or e4m3 codes plus one scale
    byte per 32 elements."""
    if wl.table_format == "e4m3":
        return wl.T * wl.K + wl.T * wl.K // 32
    return wl.T * wl.K * 2


def time_rotation(torch, layers, stream, steps, warmup, min_ms=20.0, min_samples=5):
    """Forwards rotating over the layers: `warmup` untimed steps, then a CUDA
    graph of exactly `steps` forwards, replayed until at least `min_ms` of
    replays and `min_samples` replays were timed, each replay bracketed by
    its own events on the launch stream.  Returns (median ms per step over
    the replays, steps per timed sample, the per-replay ms per step)."""
    def step(L):
        L["layer"].forward(L["hidden"], L["ids"], L.get("mask"), out=L["out"], stream=stream)

    NL = len(layers)
    for i in range(max(3, warmup)):
        step(layers[i % NL])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            step(layers[i % NL])
    graph.replay()  # the first replay uploads the graph: untimed
    torch.cuda.synchronize()
    samples = []
    total = 0.0
    while len(samples) < min_samples or total < min_ms:
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        total += ms
        samples.append(ms / steps)
        if len(samples) >= 10000:
            break
    del graph
    return statistics.median(samples), steps, samples


def time_prefetch_rotation(torch, EngramPrefetch, layers, stream, steps, warmup, min_ms=20.0,
                           min_samples=5, wkv=False):
    """The same forwards with every layer's lookup staged ahead on a side
    stream (class EngramPrefetch's start / forward / join): per group of
    the rotated layers, start() issues all their lookups (background grid)
    at once and each forward waits only for its own layer's rows, so a
    lookup runs beside the previous layers' forwards.  Captured in one CUDA
    graph of ceil(steps / layers) groups.  With wkv=True each layer's
    projection runs ahead on the side stream too (EngramPrefetch's wkv
    chain) and the forward is the gate and residual alone.  Returns (median
    ms per step, steps per sample, per-replay ms per step)."""
    NL = len(layers)
    pf = EngramPrefetch([L["layer"] for L in layers], wkv=wkv)
    groups = max(1, (steps + NL - 1) // NL)
    n = groups * NL

    def group():
        pf.start([L["ids"] for L in layers], background=True, stream=stream)
        for i, L in enumerate(layers):
            pf.forward(i, L["hidden"], None, L.get("mask"), out=L["out"], stream=stream)
        pf.join(stream=stream)

    for _ in range(max(3, warmup)):
        group()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(groups):
            group()
    graph.replay()
    torch.cuda.synchronize()
    samples, total = [], 0.0
    while len(samples) < min_samples or total < min_ms:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        total += ms
        samples.append(ms / n)
        if len(samples) >= 10000:
            break
    del graph
    pf.close()
    return statistics.median(samples), n, samples


def fp8_peak_tflops(torch, dev):
    """Dense fp8 tensor throughput of this GPU from library GEMMs (cuBLAS via
    torch._scaled_mm at 8192^3, best of 10 with CUDA events): e4m3 operands
    with per-tensor scales, and with E8M0 scales per 32 elements (the MXFP8
    form the prefill GEMM uses).  Returns {kind: TFLOP/s} for the forms this
    torch build supports."""
    M = N = K = 8192
    out = {}
    a = torch.randn(M, K, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(N, K, device=dev).to(torch.float8_e4m3fn)

    def best(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(10):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1))
        return 2.0 * M * N * K / (min(t) * 1e-3) / 1e12

    one = torch.ones((), device=dev, dtype=torch.float32)
    try:
        out["e4m3_per_tensor"] = best(
            lambda: torch._scaled_mm(a, b.t(), one, one, out_dtype=torch.bfloat16))
    except Exception as e:  # noqa: BLE001 - reported, not fatal
        out["e4m3_per_tensor_error"] = str(e).splitlines()[0][:160]
    try:
        e8 = torch.float8_e8m0fnu
        sa = torch.full((M * K // 32,), 127, dtype=torch.uint8, device=dev).view(e8)
        sb = torch.full((N * K // 32,), 127, dtype=torch.uint8, device=dev).view(e8)
        out["mxfp8_block32"] = best(
            lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16))
    except Exception as e:  # noqa: BLE001
        out["mxfp8_block32_error"] = str(e).splitlines()[0][:160]
    return out


def run_case(args):
    """W + K plain forwards of one layer: the small case for ncu captures."""
    import torch
    import __graft_entry__ as g
    import workloads as W
    from hashed_gram_engram_gb300 import Engram
    g.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    wl = W.ALL[args.case]
    wl_l, layer, _, _ = make_layer(W, Engram, wl, 0, wl.T, 0)
    st = W.make_step_inputs(wl_l, "cuda")
    out = torch.empty_like(st["hidden"])
    n = max(3, args.warmup) + args.steps
    for _ in range(n):
        layer.forward(st["hidden"], st["hash_ids"], st["token_mask"], out=out, stream=stream)
    torch.cuda.synchronize()
    err = layer.device_error()
    layer.close()
    print(json.dumps({"case": args.case, "T": wl.T, "forwards": n, "device_error": err}),
          flush=True)
    return 0 if err == 0 else 1


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.case is not None:
        return run_case(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    import __graft_entry__ as g
    import workloads as W
    from hashed_gram_engram_gb300 import (Engram, EngramPrefetch, engram_profile_enable,
                                          engram_profile_read)

    rank, local, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        g.build()
    if world > 1:
        dist.barrier()
    g.build()
    hbm_peak, bf16_peak, peak_kind = peaks()
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)

    def max_over_ranks(x):
        return reduce_max(x, world, dev)

    def rotation_layers(wl, NL, max_tokens0, table=None, seed0=0):
        out = []
        for l in range(NL):
            wl_l, layer, tab, wts = make_layer(W, Engram, wl, local,
                                               max_tokens0 if l == 0 else wl.T,
                                               seed0 + l + 1000 * rank, table=table)
            st = W.make_step_inputs(wl_l, "cuda", step=rank)
            out.append(dict(wl=wl_l, layer=layer, table=tab, wts=wts, hidden=st["hidden"],
                            ids=st["hash_ids"], mask=st["token_mask"],
                            out=torch.empty_like(st["hidden"])))
        torch.cuda.synchronize()
        return out

    # Decode: a rotation over NL independently seeded layers (each its own
    # table, wkv, q, k, hidden and ids).  Their weights (NL x 40 MiB) exceed
    # the 129 MB L2, so consecutive steps read weights from HBM and no flush
    # is needed between them.  The rotation is captured in a CUDA graph (as a
    # serving engine runs decode) and replayed.
    wl = W.DECODE
    NL = args.layers
    layers = rotation_layers(wl, NL, W.PREFILL.T)
    clocks = Clocks(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    ms_step, steps, samples = time_rotation(torch, layers, stream, args.steps, args.warmup,
                                            args.min_ms)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_step = max_over_ranks(ms_step)
    value = world * wl.T / (ms_step * 1e-3)
    step_bytes = algorithmic_bytes(wl)
    # one kernel per step: its average duration is the step time (launch gaps included)
    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    traffic = stored_traffic(DECODE_PROFILE, DECODE_SOURCES)

    # single-step latency with L2 flushed before the step (cold code, page
    # tables and weights), and the kernel's own event time
    L0 = layers[0]

    def step0():
        L0["layer"].forward(L0["hidden"], L0["ids"], None, out=L0["out"], stream=stream)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    lat = []
    engram_profile_enable(L0["layer"].handle, 1)
    kern = []
    for i in range(min(args.steps, 200)):
        flush.zero_()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        step0()
        a1.record(stream)
        kern.append(engram_profile_read(L0["layer"].handle)[1])
        torch.cuda.synchronize()
        lat.append(a0.elapsed_time(a1))
    engram_profile_enable(L0["layer"].handle, 0)
    del flush

    # end to end through the host-buffer entry points, rotating over the
    # layers like the device timing: every step copies its hidden and ids
    # from pinned host memory and its output back.  engram_forward_host runs
    # a step's copies and forward in order; engram_forward_host_pipelined
    # (the figure reported) lets a step's input copy overlap the previous
    # step's forward and output copy.
    host_in = [(L["hidden"].cpu().pin_memory(), L["ids"].cpu().pin_memory()) for L in layers]
    hid_h, ids_h = host_in[0]
    out_h = torch.empty_like(hid_h).pin_memory()
    ne = min(args.steps, 500)

    def e2e_ms_per_step(mode):
        def fwd(i):
            L = layers[i % NL]["layer"]
            hid, ids = host_in[i % NL]
            if mode == "serial":
                L.forward_host(hid, ids, None, out_h, stream=stream)
            else:
                L.forward_host_pipelined(hid, ids, None, out_h, stream=stream,
                                         defer_output=mode == "deferred")

        def flush():
            if mode == "deferred":
                for L in layers:
                    L["layer"].flush_host(stream)
        for i in range(3 * NL):
            fwd(i)
        flush()
        torch.cuda.synchronize()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for i in range(ne):
            fwd(i)
        flush()  # every step's output copy inside the timed region
        b1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(b0.elapsed_time(b1) / ne)

    e2e_ms = e2e_ms_per_step("deferred")
    e2e_ordered_ms = e2e_ms_per_step("pipelined")
    e2e_serial_ms = e2e_ms_per_step("serial")

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {**decode_config(wl),
                   "layers_rotated": NL,
                   "seeds": {"layers": [int(L["wl"].seed) for L in layers],
                             "generator": "torch.Generator.manual_seed per tensor kind"},
                   "l2": f"inputs larger than L2: {NL} layers' weights ({NL * 40} MiB) rotated",
                   "timing": f"CUDA graph of exactly {steps} steps (--steps), replayed "
                             f"{len(samples)}x, each replay timed by CUDA events on the launch "
                             f"stream; value from the median replay",
                   "replay_ms_per_step": {"min": min(samples), "median": ms_step,
                                          "max": max(samples)},
                   "parallelism": f"replicas x{world} (token-sharded, no collective)"},
        "roofline": {"bound": "hbm",
                     "kernel": "decode_fused_kernel (gather + tcgen05 wkv + gate, one launch)",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_kind": peak_kind, "algorithmic_bytes": step_bytes,
                     "kernel_ms": ms_step},
        "latency_l2_flushed_us": {"step_median": 1e3 * float(np.median(lat)),
                                  "kernel_median": 1e3 * float(np.median(kern))},
        "e2e": {"value": world * wl.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(hid_h.numel() * 2 + ids_h.numel() * 4),
                "d2h_bytes_per_step": int(out_h.numel() * 2),
                "ms_per_step": e2e_ms, "steps": ne,
                "how": f"engram_forward_host_pipelined with ENGRAM_HOST_DEFER_OUTPUT, {ne} "
                       f"back-to-back steps rotating over {NL} layers (a step's input copy "
                       f"overlaps the previous step, its output copy the next one), then "
                       f"engram_forward_host_flush; CUDA events around all of it",
                "ordered_value": world * wl.T / (e2e_ordered_ms * 1e-3),
                "ordered_how": "engram_forward_host_pipelined: the stream waits for each "
                               "step's output copy before the next step",
                "serial_value": world * wl.T / (e2e_serial_ms * 1e-3),
                "serial_how": "engram_forward_host: each step's copies and forward in order"},
        "gpu_launches": steps * len(samples),
        "gpu_launches_per_step": 1,
        "clocks": clk,
    }
    launches = steps * len(samples)

    def prefill_block(layer, pw, kernel_name, peak, peak_name, tile_cols):
        """Per-step time of a prefill forward and its kernels' event times."""
        pstep = W.make_step_inputs(pw, "cuda", step=rank)
        ph, pids, pmask = pstep["hidden"], pstep["hash_ids"], pstep["token_mask"]
        pout = torch.empty_like(ph)
        pf = lambda: layer.forward(ph, pids, pmask, out=pout, stream=stream)  # noqa: E731
        for _ in range(3):
            pf()
        torch.cuda.synchronize()
        pk = max(5, min(50, args.steps))
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(pk):
            pf()
        c1.record(stream)
        torch.cuda.synchronize()
        p_ms = max_over_ranks(c0.elapsed_time(c1) / pk)
        engram_profile_enable(layer.handle, 1)
        pprof = []
        for _ in range(10):
            pf()
            pprof.append(engram_profile_read(layer.handle))
        engram_profile_enable(layer.handle, 0)
        pprof = np.array(pprof)
        pw_ms = float(np.median(pprof[:, 1]))
        flops = 2.0 * pw.T * pw.N * pw.K
        tf = flops / (pw_ms * 1e-3) / 1e12
        gate_ms = float(np.median(pprof[:, 2]))
        gb = gate_ring_bytes(pw, tile_cols)
        return pk * 3 + 30, {
            "workload": pw.name, "T": pw.T, "tokens_per_s": world * pw.T / (p_ms * 1e-3),
            "ms_per_step": p_ms, "l2": "inputs larger than L2 (hidden "
                                      f"{pw.T * pw.hc_mult * pw.dim * 2 >> 20} MiB per step)",
            "kernel_ms": {"gather": float(np.median(pprof[:, 0])), "wkv": pw_ms,
                          "gate": float(np.median(pprof[:, 2]))},
            "roofline": {"bound": "tensor", "kernel": kernel_name, "achieved": tf,
                         "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_kind": peak_name,
                         "traffic": stored_traffic(profile_path("wkv_gemm_kernel", pw),
                                                   GEMM_SOURCES)},
            "gate_roofline": {"bound": "hbm", "kernel": "gate_ring_kernel",
                              "achieved": gb / (gate_ms * 1e-3) / 1e9, "peak": hbm_peak,
                              "unit": "GB/s", "frac": gb / (gate_ms * 1e-3) / 1e9 / hbm_peak,
                              "algorithmic_bytes": gb, "peak_kind": peak_kind,
                              "traffic": stored_traffic(profile_path("gate_ring_kernel", pw),
                                                        GATE_SOURCES)},
        }

    if not args.no_prefill:
        n, line["prefill"] = prefill_block(
            L0["layer"], W.PREFILL, "wkv_gemm_kernel<bf16> (CTA pairs, cta_group::2)", bf16_peak,
            peak_kind, 256)
        launches += n

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = dict(table=W.bits(L0["table"]), row_offset=W.row_offsets(wl.rows),
                    rows=np.asarray(wl.rows, np.int64), wkv=W.bits(L0["wts"]["wkv"]),
                    q=W.bits(L0["wts"]["q_weight"]), k=W.bits(L0["wts"]["k_weight"]))
        inp = dict(hidden=W.bits(L0["hidden"]), ids=L0["ids"].cpu().numpy(), mask=None)
        tps, n, el = cpu_oracle_tokens_per_s(wl, host, inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} decode-step tokens ({el:.1f} s, "
                                          f"single-threaded fp64 C oracle)",
                                "host_cores": os.cpu_count()}
    for L in layers:
        L["layer"].close()
    del layers, L0

    if not args.no_mxfp8:
        # MXFP8 wkv: the same decode rotation (T = 64, D = 7168) and the
        # T = 4096 prefill step on the first layer
        mw = W.MXFP8_DECODE
        mlayers = rotation_layers(mw, NL, W.MXFP8_PREFILL.T, seed0=50)
        m_ms, m_steps, m_samp = time_rotation(torch, mlayers, stream, args.steps, args.warmup,
                                              args.min_ms)
        m_ms = max_over_ranks(m_ms)
        mb = algorithmic_bytes(mw)
        line["mxfp8_decode"] = {
            "workload": mw.name, "T": mw.T, "dim": mw.dim, "tokens_per_s": world * mw.T / (m_ms * 1e-3),
            "ms_per_step": m_ms, "steps": m_steps, "layers_rotated": NL,
            "wkv": f"e4m3 [{mw.N}, {mw.K}] + E8M0 [{mw.N // 32}, {mw.K // 32}]",
            "l2": f"inputs larger than L2: {NL} layers' weights ({NL * mw.N * mw.K >> 20} MiB)",
            "roofline": {"bound": "hbm", "kernel": "decode_fused_kernel<mxfp8>",
                         "achieved": mb / (m_ms * 1e-3) / 1e9, "peak": hbm_peak,
                         "unit": "GB/s", "frac": mb / (m_ms * 1e-3) / 1e9 / hbm_peak,
                         "algorithmic_bytes": mb, "peak_kind": peak_kind},
        }
        launches += m_steps * len(m_samp)
        if not args.no_prefill:
            # the fp8 tensor peak this GPU reaches with library GEMMs: the
            # MXFP8 (E8M0 per 32) form when the torch build has it, else
            # per-tensor e4m3, else 2 x the measured bf16 peak (nominal ratio)
            fp8 = fp8_peak_tflops(torch, dev)
            if "mxfp8_block32" in fp8:
                fp8_peak, fp8_kind = fp8["mxfp8_block32"], "measured: cuBLAS MXFP8 GEMM 8192^3"
            elif "e4m3_per_tensor" in fp8:
                fp8_peak, fp8_kind = fp8["e4m3_per_tensor"], "measured: cuBLAS e4m3 GEMM 8192^3"
            else:
                fp8_peak, fp8_kind = 2.0 * bf16_peak, f"{peak_kind} bf16 x 2 (nominal ratio)"
            line["fp8_peak_measured"] = fp8
            mxp = W.MXFP8_PREFILL
            n, line["mxfp8_prefill"] = prefill_block(
                mlayers[0]["layer"], mxp, "wkv_gemm_kernel<mxfp8> (CTA pairs, cta_group::2)",
                fp8_peak, fp8_kind, 224 if mxp.dim % 224 == 0 else 128)
            launches += n
        for L in mlayers:
            L["layer"].close()
        del mlayers

    def offload_line(ow, seed0):
        """The offload step: the table in pinned host memory, shared by the
        rotated layers; every gathered row crosses the host link."""
        fp8 = ow.table_format == "e4m3"
        need = ow.total_rows * ow.head_dim * (1 + 1 / 32 if fp8 else 2)
        avail = W.host_memory_bytes()
        if avail is not None and avail < need + (8 << 30):
            return {"workload": ow.name, "skipped":
                    f"{int(need) >> 30} GiB pinned table, {avail >> 30} GiB host memory free"}, 0
        otable = (W.make_table(ow, "cuda"), W.make_table_scale(ow, "cuda"))
        olayers = rotation_layers(ow, 4, ow.T, table=otable, seed0=seed0)
        o_ms, o_steps, o_samp = time_rotation(torch, olayers, stream, args.steps, args.warmup,
                                              args.min_ms)
        o_ms = max_over_ranks(o_ms)
        # the same rotation with each layer's host-table lookup staged ahead
        # on a side stream, beside the previous layers' forwards
        p_ms, p_steps, p_samp = time_prefetch_rotation(torch, EngramPrefetch, olayers, stream,
                                                       args.steps, args.warmup, args.min_ms)
        p_ms = max_over_ranks(p_ms)
        k_ms, k_steps, k_samp = time_prefetch_rotation(torch, EngramPrefetch, olayers, stream,
                                                       args.steps, args.warmup, args.min_ms,
                                                       wkv=True)
        k_ms = max_over_ranks(k_ms)
        ob = algorithmic_bytes(ow)
        host_b = row_bytes(ow)
        kind = "e4m3 codes + ue8m0 scales per 32" if fp8 else "bf16"
        res = {
            "workload": ow.name, "T": ow.T, "tokens_per_s": world * ow.T / (o_ms * 1e-3),
            "ms_per_step": o_ms, "steps": o_steps, "layers_rotated": 4,
            "table": f"{need / 1e9:.2f} GB {kind} in pinned host memory",
            "host_link": {"bytes_per_step": host_b,
                          "GB_per_s": host_b / (o_ms * 1e-3) / 1e9,
                          "rows_per_step": ow.T * ow.n_hash_cols},
            "roofline": {"bound": "hbm", "kernel": "decode_fused_kernel (host table)",
                         "achieved": ob / (o_ms * 1e-3) / 1e9, "peak": hbm_peak,
                         "unit": "GB/s", "frac": ob / (o_ms * 1e-3) / 1e9 / hbm_peak,
                         "algorithmic_bytes": ob, "peak_kind": peak_kind},
            "prefetched": {
                "how": "EngramPrefetch: all layers' lookups (background grid) on a side stream "
                       "at start, each forward waits for its own rows only",
                "tokens_per_s": world * ow.T / (p_ms * 1e-3), "ms_per_step": p_ms,
                "steps": p_steps,
                "host_link_GB_per_s": host_b / (p_ms * 1e-3) / 1e9,
                "roofline_frac": ob / (p_ms * 1e-3) / 1e9 / hbm_peak},
            "prefetched_wkv": {
                "how": "EngramPrefetch(wkv=True): each layer's gather and projection (the fused "
                       "kernel writing bf16 kv) on the side stream, the forward is "
                       "engram_gate_noalloc over that kv",
                "tokens_per_s": world * ow.T / (k_ms * 1e-3), "ms_per_step": k_ms,
                "steps": k_steps, "roofline_frac": ob / (k_ms * 1e-3) / 1e9 / hbm_peak},
        }
        for L in olayers:
            L["layer"].close()
        del olayers, otable
        return res, o_steps * len(o_samp) + p_steps * len(p_samp) * 2 + k_steps * len(k_samp) * 2

    if not args.no_offload:
        line["offload"], n = offload_line(W.OFFLOAD, 70)
        launches += n

    if not args.no_e4m3_table:
        # fp8 tables (the pages' storage): the decode rotation and the
        # offload step with e4m3 rows and ue8m0 scales, dequantized by the gather
        ew = W.DECODE_E4M3
        elayers = rotation_layers(ew, NL, ew.T, seed0=90)
        e_ms, e_steps, e_samp = time_rotation(torch, elayers, stream, args.steps, args.warmup,
                                              args.min_ms)
        e_ms = max_over_ranks(e_ms)
        eb = algorithmic_bytes(ew)
        line["decode_e4m3_table"] = {
            "workload": ew.name, "T": ew.T, "tokens_per_s": world * ew.T / (e_ms * 1e-3),
            "ms_per_step": e_ms, "steps": e_steps, "layers_rotated": NL,
            "table": f"{ew.total_rows * ew.head_dim * (1 + 1 / 32) / 1e9:.2f} GB e4m3 + ue8m0 "
                     f"per layer in HBM",
            "roofline": {"bound": "hbm", "kernel": "decode_fused_kernel (e4m3 table)",
                         "achieved": eb / (e_ms * 1e-3) / 1e9, "peak": hbm_peak,
                         "unit": "GB/s", "frac": eb / (e_ms * 1e-3) / 1e9 / hbm_peak,
                         "algorithmic_bytes": eb, "peak_kind": peak_kind},
        }
        launches += e_steps * len(e_samp)
        for L in elayers:
            L["layer"].close()
        del elayers
        if not args.no_offload:
            line["offload_e4m3_table"], n = offload_line(W.OFFLOAD_E4M3, 110)
            launches += n

    line["gpu_launches_all_timed_regions"] = launches
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
