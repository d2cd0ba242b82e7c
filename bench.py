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
too.

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
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--layers", type=int, default=6)
    p.add_argument("--case", choices=["decode", "prefill"], default=None,
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
    # size the per-step sample so that warmup + steps take about 90 s
    per_tok, _, _ = cpu_oracle_tokens_per_s(wl, host, inp, 0.0, max_tokens=1)
    budget = 90.0 / max(1, args.steps + args.warmup)
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
        "config": {"workload": wl.name, "T": wl.T, "dim": wl.dim, "hc_mult": wl.hc_mult,
                   "n_hash_cols": wl.n_hash_cols, "head_dim": wl.head_dim,
                   "wkv": "bf16 [20480, 1024]", "tokens_per_step_sample": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} of the {wl.T} decode-step tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def source_digest(names):
    """sha256 (12 hex) of kernel sources, to tell whether a stored ncu
    figure still describes the kernel that runs."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "hashed_gram_engram_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


DECODE_SOURCES = ("decode_fused.cu", "ptx.cuh", "internal.h")
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_fused_kernel_decode_T64.md")


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


def make_layer(W, Engram, wl, device_index, max_tokens, layer_seed):
    import dataclasses
    wl_l = dataclasses.replace(wl, seed=wl.seed + 101 * layer_seed)
    table = W.make_table(wl_l, "cuda")
    wts = W.make_weights(wl_l, "cuda")
    layer = Engram(dim=wl.dim, hc_mult=wl.hc_mult, max_ngram_size=wl.max_ngram_size,
                   n_heads=wl.n_heads, head_dim=wl.head_dim, max_tokens=max_tokens,
                   table=table, rows=wl.rows, row_offset=W.row_offsets(wl.rows),
                   wkv=wts["wkv"], q_weight=wts["q_weight"], k_weight=wts["k_weight"],
                   eps=wl.eps, clamp=wl.clamp, device=device_index)
    return wl_l, layer, table, wts


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
    wl = W.DECODE if args.case == "decode" else W.PREFILL
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
    from hashed_gram_engram_gb300 import Engram, engram_profile_enable, engram_profile_read

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

    # Decode: a rotation over NL independently seeded layers (each its own
    # table, wkv, q, k, hidden and ids).  Their packed weights (NL x 40 MiB)
    # exceed the 129 MB L2, so consecutive steps read weights from HBM and no
    # flush is needed between them.  The rotation is captured in a CUDA graph
    # (as a serving engine runs decode) and replayed.
    wl = W.DECODE
    NL = args.layers
    layers = []
    for l in range(NL):
        wl_l, layer, table, wts = make_layer(W, Engram, wl, local, W.PREFILL.T if l == 0 else wl.T,
                                             l + 1000 * rank)
        st = W.make_step_inputs(wl_l, "cuda", step=rank)
        layers.append(dict(wl=wl_l, layer=layer, table=table, wts=wts, hidden=st["hidden"],
                           ids=st["hash_ids"], out=torch.empty_like(st["hidden"])))
    torch.cuda.synchronize()

    def step(L):
        L["layer"].forward(L["hidden"], L["ids"], None, out=L["out"], stream=stream)

    for _ in range(max(3, args.warmup)):
        for L in layers:
            step(L)
    torch.cuda.synchronize()
    per_graph = NL * max(1, 24 // NL)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(per_graph):
            step(layers[i % NL])
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    replays = max(1, args.steps // per_graph)
    steps = replays * per_graph

    clocks = Clocks(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = e0.elapsed_time(e1)
    t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms = float(t.item())
    ms_step = total_ms / steps
    value = world * wl.T * steps / (total_ms / 1e3)

    step_bytes = (wl.N * wl.K * 2 + 2 * wl.T * wl.hc_mult * wl.dim * 2 + wl.T * wl.K * 2
                  + wl.T * wl.n_hash_cols * 4 + 2 * wl.hc_mult * wl.dim * 2)
    # one kernel per step: its average duration is the step time (launch gaps included)
    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    traffic = stored_traffic(DECODE_PROFILE, DECODE_SOURCES)

    # single-step latency with L2 flushed before the step (cold code, page
    # tables and weights), and the kernel's own event time
    L0 = layers[0]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    lat = []
    engram_profile_enable(L0["layer"].handle, 1)
    kern = []
    for i in range(min(args.steps, 200)):
        flush.zero_()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        step(L0)
        a1.record(stream)
        kern.append(engram_profile_read(L0["layer"].handle)[1])
        torch.cuda.synchronize()
        lat.append(a0.elapsed_time(a1))
    engram_profile_enable(L0["layer"].handle, 0)
    del flush

    # end to end through the host-buffer entry point
    hid_h = L0["hidden"].cpu().pin_memory()
    ids_h = L0["ids"].cpu().pin_memory()
    out_h = torch.empty_like(hid_h).pin_memory()
    fwd_h = lambda: L0["layer"].forward_host(hid_h, ids_h, None, out_h, stream=stream)  # noqa: E731
    for _ in range(3):
        fwd_h()
    torch.cuda.synchronize()
    ne = min(args.steps, 500)
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(ne):
        fwd_h()
    b1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = b0.elapsed_time(b1) / ne
    th = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(th, op=dist.ReduceOp.MAX)
    e2e_ms = float(th.item())

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "decode", "T": wl.T, "dim": wl.dim, "hc_mult": wl.hc_mult,
                   "n_hash_cols": wl.n_hash_cols, "head_dim": wl.head_dim,
                   "table_rows": wl.total_rows, "wkv": "bf16 [20480, 1024]", "mask": None,
                   "layers_rotated": NL,
                   "l2": f"inputs larger than L2: {NL} layers' weights ({NL * 40} MiB) rotated",
                   "timing": f"CUDA graph of {per_graph} steps replayed {replays}x, events on "
                             "the launch stream",
                   "parallelism": f"replicas x{world} (token-sharded, no collective)"},
        "roofline": {"bound": "hbm",
                     "kernel": "decode_fused_kernel (gather4 + tcgen05 wkv + gate, one launch)",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_kind": peak_kind, "algorithmic_bytes": step_bytes,
                     "kernel_ms": ms_step},
        "latency_l2_flushed_us": {"step_median": 1e3 * float(np.median(lat)),
                                  "kernel_median": 1e3 * float(np.median(kern))},
        "e2e": {"value": wl.T / (e2e_ms * 1e-3) * world, "unit": "tokens/s",
                "h2d_bytes_per_step": int(hid_h.numel() * 2 + ids_h.numel() * 4),
                "d2h_bytes_per_step": int(out_h.numel() * 2)},
        "gpu_launches": steps,
        "clocks": clk,
    }

    if not args.no_prefill:
        pw = W.PREFILL
        layer = L0["layer"]
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
        p_ms = c0.elapsed_time(c1) / pk
        engram_profile_enable(layer.handle, 1)
        pprof = []
        for _ in range(10):
            pf()
            pprof.append(engram_profile_read(layer.handle))
        engram_profile_enable(layer.handle, 0)
        pprof = np.array(pprof)
        pw_ms = float(np.median(pprof[:, 1]))
        flops = 2.0 * pw.T * pw.N * pw.K
        line["prefill"] = {
            "workload": "prefill", "T": pw.T, "tokens_per_s": pw.T / (p_ms * 1e-3),
            "ms_per_step": p_ms, "l2": "inputs larger than L2 (hidden 256 MiB per step)",
            "kernel_ms": {"gather": float(np.median(pprof[:, 0])), "wkv": pw_ms,
                          "gate": float(np.median(pprof[:, 2]))},
            "roofline": {"bound": "tensor", "kernel": "wkv_gemm_bf16 (token-as-M)",
                         "achieved": flops / (pw_ms * 1e-3) / 1e12, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": flops / (pw_ms * 1e-3) / 1e12 / bf16_peak,
                         "peak_kind": peak_kind},
        }

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
    if rank == 0:
        print(json.dumps(line), flush=True)
    for L in layers:
        L["layer"].close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
