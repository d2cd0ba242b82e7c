"""Shared helpers of the GPU parity tests: build a layer from a workload,
run it through the C ABI, run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import oracle_pool
import workloads as W
from hashed_gram_engram_gb300 import Engram


def np_bf16(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def oracle_all(case, inp, quantize_act=False, workers=None):
    """Oracle outputs for every token of a large step: the gather in this
    process, then wkv and the gate over token chunks in spawned worker
    processes, one single-threaded oracle each (the host's cores in
    parallel).  Returns rows, out_f64, out_bf16, gate and value (the last D
    kv columns; the keys are not kept)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os
    import tempfile
    hs = case.host()
    wl = case.wl
    ids = inp["hash_ids"].cpu().numpy()
    if hs["table_scale"] is None:
        rows, nbad = oracle.gather(hs["table"], case.row_offset, case.rows, ids, wl.head_dim)
    else:
        rows, nbad = oracle.gather_e4m3(hs["table"], hs["table_scale"], case.row_offset,
                                        case.rows, ids, wl.head_dim)
    hidden = W.bits(inp["hidden"])
    mask = None if inp["token_mask"] is None else W.bits(inp["token_mask"])
    T = hidden.shape[0]
    workers = workers or max(1, min(32, os.cpu_count() or 1))
    bounds = np.linspace(0, T, workers * 2 + 1).astype(int)
    with tempfile.TemporaryDirectory() as d:
        w_path = os.path.join(d, "w.npy")
        np.save(w_path, hs["wkv"])
        jobs = [(rows[a:b], w_path, hs["wkv_scale"], hidden[a:b], hs["q"], hs["k"],
                 None if mask is None else mask[a:b], wl.eps, wl.clamp, quantize_act,
                 wl.hc_mult, wl.dim) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        with cf.ProcessPoolExecutor(max_workers=workers,
                                    mp_context=mp.get_context("spawn")) as ex:
            parts = list(ex.map(oracle_pool.oracle_chunk, jobs))
    ref = {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}
    ref.update(rows=rows, n_bad=nbad)
    return ref


class Case:
    """A workload's weights on the GPU plus its host copies for the oracle."""

    def __init__(self, wl: W.Workload, max_tokens=None, gen_device=None):
        self.wl = wl
        dev = torch.device("cuda", 0)
        small = wl.total_rows * wl.head_dim < (1 << 24)
        gen = gen_device or ("cpu" if small else "cuda")
        table = W.make_table(wl, gen)
        tscale = W.make_table_scale(wl, gen)
        if wl.table_location == "device":
            table = table.to(dev)
            tscale = None if tscale is None else tscale.to(dev)
        self.table_scale = tscale
        wts = W.make_weights(wl, gen)
        self.table = table
        self.wkv = wts["wkv"].to(dev)
        self.wkv_scale = None if wts["wkv_scale"] is None else wts["wkv_scale"].to(dev)
        self.q = wts["q_weight"].to(dev)
        self.k = wts["k_weight"].to(dev)
        self.rows = np.asarray(wl.rows, np.int64)
        self.row_offset = W.row_offsets(wl.rows)
        self.gen = gen
        self.layer = Engram(dim=wl.dim, hc_mult=wl.hc_mult, max_ngram_size=wl.max_ngram_size,
                            n_heads=wl.n_heads, head_dim=wl.head_dim,
                            max_tokens=max_tokens or wl.T, table=self.table, rows=self.rows,
                            row_offset=self.row_offset, wkv=self.wkv, wkv_scale=self.wkv_scale,
                            q_weight=self.q, k_weight=self.k, eps=wl.eps, clamp=wl.clamp,
                            device=0, keep_value=True, table_scale=self.table_scale)
        self._host = None

    def host(self):
        if self._host is None:
            self._host = dict(
                table=W.bits(self.table),
                table_scale=None if self.table_scale is None else W.bits(self.table_scale),
                wkv=W.bits(self.wkv),
                wkv_scale=None if self.wkv_scale is None else W.bits(self.wkv_scale),
                q=W.bits(self.q), k=W.bits(self.k))
        return self._host

    def step_inputs(self, T=None, step=0):
        d = W.make_step_inputs(self.wl, self.gen, T, step)
        dev = torch.device("cuda", 0)
        return {k: (None if v is None else v.to(dev)) for k, v in d.items()}

    def oracle(self, inp, tokens=None, quantize_act=False):
        """Oracle outputs for all tokens, or for the listed token indices."""
        hs = self.host()
        hidden = W.bits(inp["hidden"])
        ids = inp["hash_ids"].cpu().numpy()
        mask = None if inp["token_mask"] is None else W.bits(inp["token_mask"])
        if tokens is not None:
            hidden, ids = hidden[tokens], np.ascontiguousarray(ids[tokens])
            mask = None if mask is None else mask[tokens]
        return oracle.forward(hs["table"], self.row_offset, self.rows, ids, self.wl.head_dim,
                              hs["wkv"], hidden, hs["q"], hs["k"], mask, Ws=hs["wkv_scale"],
                              eps=self.wl.eps, clamp=self.wl.clamp, quantize_act=quantize_act,
                              table_scale=hs["table_scale"])


def compare(case: Case, inp, out, ref, tokens=None, gate=None, value=None, tol=None,
            value_rtol=1e-2, gate_rtol=1e-2, rounding=True):
    """Asserts the parity bar; returns a dict of the errors seen.  With
    rounding=False the rounding-level bound is skipped (a reference that
    differs from the kernel by more than rounding, e.g. unquantised MXFP8
    activations)."""
    wl = case.wl
    tol = wl.tol if tol is None else tol
    got_bits = W.bits(out)
    hid_bits = W.bits(inp["hidden"])
    if tokens is not None:
        got_bits, hid_bits = got_bits[tokens], hid_bits[tokens]
    got = np_bf16(got_bits)
    exp = ref["out_f64"]
    err = float(np.abs(got - exp).max()) if got.size else 0.0
    assert err <= tol, f"max abs err {err} > {tol}"
    # rounding-level agreement: the only differences left are the fp32
    # projection, the bf16 value of the token-as-M path and the final RTNE
    value_ref = ref["value"] if "value" in ref else ref["kv"][:, wl.hc_mult * wl.dim:]
    bound = 2.0 ** -8 * np.abs(exp) + 2.0 ** -8 * np.abs(value_ref)[:, None, :] + 1e-5
    if rounding:
        assert np.all(np.abs(got - exp) <= bound), "output differs beyond rounding level"
    res = dict(max_abs_err=err)
    mask = inp["token_mask"]
    if mask is not None:
        m = W.bits(mask).astype(bool)
        if tokens is not None:
            m = m[tokens]
        assert np.array_equal(got_bits[~m], hid_bits[~m]), "masked rows differ from hidden"
    if gate is not None:
        g = gate.cpu().numpy().astype(np.float64)
        if tokens is not None:
            g = g[tokens]
        gerr = float(np.abs(g - ref["gate"]).max() / max(np.abs(ref["gate"]).max(), 1e-30))
        assert gerr <= gate_rtol, f"gate rel err {gerr}"
        res["gate_rel_err"] = gerr
    if value is not None:
        v = value.cpu().numpy().astype(np.float64)
        if tokens is not None:
            v = v[tokens]
        verr = float(np.abs(v - value_ref).max() / max(np.abs(value_ref).max(), 1e-30))
        assert verr <= value_rtol, f"value rel err {verr}"
        res["value_rel_err"] = verr
    return res
