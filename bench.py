#!/usr/bin/env python
"""Benchmark: FP8 paged decode attention step — achieved HBM GB/s and µs/step vs bf16.

One step = one decode step of every layer of the workload: for each layer the new
token's K/V are written into the paged cache (e4m3 with per-KV-head scales) and the
decode attention reads the whole cached context (split-K + FP32 merge), both in one
launch (fp8_decode_step) — on bf16 layers too, so that the FP8 and BF16 steps have the
same launch structure.
Inputs are seeded synthetic tensors shaped like the pages' Llama-3.1-8B decode under
load (32 layers, 32/8 heads, head_dim 128, batch 8, contexts U[16384, 24576]); the
cache (10.5 GB per step) is far larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2] [--impl reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 paged decode attn: achieved HBM GB/s (% of peak) and µs/step vs bf16"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- helpers

def _env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C++/CUDA source without its comments, trailing blanks and empty lines."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def _local_includes(csrc: str, name: str, seen=None) -> set:
    """The files of csrc/ that `name` includes, directly or through one another."""
    import re
    seen = set() if seen is None else seen
    path = os.path.join(csrc, name)
    if name in seen or not os.path.exists(path):
        return seen
    seen.add(name)
    for inc in re.findall(r'^\s*#include\s+"([^"/]+)"', open(path, encoding="utf-8").read(), flags=re.M):
        _local_includes(csrc, inc, seen)
    return seen


def kernel_source_sha(kernel_file: str) -> str:
    """First 16 hex digits of the sha256 of the code (comments removed) of a kernel's .cu
    file followed by those of the shared headers common.cuh, tc.cuh, decode_common.cuh and
    kernels.h (in that order) that it includes: a profile summary stays valid only while
    none of them has changed."""
    csrc = os.path.join(ROOT, "fp8_kv_cache_quant_gb300", "csrc")
    used = _local_includes(csrc, kernel_file)
    h = hashlib.sha256()
    for name in (kernel_file, "common.cuh", "tc.cuh", "decode_common.cuh", "kernels.h"):
        if name in used:
            h.update(_code_only(open(os.path.join(csrc, name), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def _traffic_record(kernel_file: str, summary: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source (same sha256); else None."""
    path = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "fp8_kv_cache_quant_gb300", "csrc", kernel_file)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    sha = kernel_source_sha(kernel_file)
    rec = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    if rec.get("source_sha256_16") != sha:
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed regions run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

def decode_bytes(w, ctx, layer_is_bf16):
    """Algorithmic HBM bytes of one step: every cached key/value of every layer read once,
    Q read, O written, block-table entries read, the new token's bf16 K/V read and its
    cache bytes written.  Split-K partials are overhead and excluded."""
    import numpy as np
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    per_layer = []
    for l in range(w.num_layers):
        S = 2 if layer_is_bf16[l] else 1
        win = w.layer_window(l)
        teff = [min(int(t), win) if win else int(t) for t in ctx]
        kv = sum(2 * Hkv * D * S * t for t in teff)
        table = sum(4 * ((t + 15) // 16 + 1) for t in teff)
        qo = 2 * B * Hq * D * 2
        write = B * Hkv * D * (2 * 2 + 2 * S)
        per_layer.append({"kv": kv, "decode": kv + table + qo, "write": write})
    return per_layer


class DecodeState:
    def __init__(self, f, w, device, all_bf16=False, no_skip=False):
        import numpy as np
        import torch
        import synth
        self.w = w
        self.f = f
        self.ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
        self.table, self.nb = synth.block_table(self.ctx, seed=w.seed)
        if all_bf16:
            self.mask = np.ones(w.num_layers, np.uint8)
        elif no_skip:
            self.mask = np.zeros(w.num_layers, np.uint8)
        else:
            self.mask = w.skip_mask()
        self.bf16 = [bool(x) for x in self.mask]
        # every layer writes the current token and decodes in one launch (fp8_decode_step)
        self.fusable = [True for _ in self.bf16]
        self.gran = f.SCALE_PER_HEAD if w.scale_mode == "amax" else f.SCALE_PER_TENSOR
        self.table_d = torch.from_numpy(self.table).to(device)
        self.ctx_d = torch.from_numpy(self.ctx).to(device)
        cu = np.concatenate([[0], np.cumsum(self.ctx)])
        last = cu[1:] - 1
        self.slots_new = torch.from_numpy(synth.slot_mapping(self.table, self.ctx, positions=[[int(t) - 1] for t in self.ctx])).to(device)
        slots_all = torch.from_numpy(synth.slot_mapping(self.table, self.ctx)).to(device)
        self.layers = []
        max_ws = 0
        L, B, Hq, Hkv, D = w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
        # one contiguous buffer per kind for all layers: a step's inputs and outputs move
        # between host and device in one copy each
        self.q_all = torch.empty((L, B, Hq, D), dtype=torch.bfloat16, device=device)
        self.k_all = torch.empty((L, B, Hkv, D), dtype=torch.bfloat16, device=device)
        self.v_all = torch.empty((L, B, Hkv, D), dtype=torch.bfloat16, device=device)
        self.out_all = torch.empty((L, B, Hq, D), dtype=torch.bfloat16, device=device)
        idx = torch.from_numpy(last).to(device)
        for l in range(L):
            data = synth.decode_layer(w, l, self.ctx, device=device)
            cache = f.LayerCache.empty(self.nb, Hkv, D, bf16=self.bf16[l], device=device)
            f.kv_quant_cache(data.k, data.v, slots_all, cache, data.k_scale, data.v_scale, self.gran, layer=l,
                             skip_layer_mask=self.mask)
            self.q_all[l].copy_(data.q)
            self.k_all[l].copy_(data.k[idx])
            self.v_all[l].copy_(data.v[idx])
            lay = dict(cache=cache, q=self.q_all[l], k_new=self.k_all[l], v_new=self.v_all[l],
                       qs=data.q_scale, ks=data.k_scale, vs=data.v_scale, window=w.layer_window(l),
                       out=self.out_all[l])
            self.layers.append(lay)
            max_ws = max(max_ws, f.fp8_decode_attn_workspace_size(B, Hq, Hkv, D, self.table.shape[1],
                                                                  lay["window"]))
            del data
        torch.cuda.synchronize()
        self.ws = torch.zeros(max_ws, dtype=torch.uint8, device=device)   # split counters start at zero
        self.bytes = decode_bytes(w, self.ctx, self.bf16)

    def step(self, decode_only=False, fused=True):
        """One decode step over all layers: each layer's current-token cache write and its
        decode attention, in one launch (fp8_decode_step, e4m3 layers) or two (kv_quant_cache
        then fp8_decode_attn); decode_only leaves the writes out."""
        f = self.f
        for l, lay in enumerate(self.layers):
            kw = dict(window=lay["window"], layer=l, skip_layer_mask=self.mask, out=lay["out"], workspace=self.ws)
            if not decode_only and fused and self.fusable[l]:
                f.fp8_decode_step(lay["k_new"], lay["v_new"], lay["q"], lay["cache"], self.table_d, self.ctx_d,
                                  lay["qs"], lay["ks"], lay["vs"], self.gran, **kw)
                continue
            if not decode_only:
                f.kv_quant_cache(lay["k_new"], lay["v_new"], self.slots_new, lay["cache"], lay["ks"], lay["vs"],
                                 self.gran, layer=l, skip_layer_mask=self.mask)
            f.fp8_decode_attn(lay["q"], lay["cache"], self.table_d, self.ctx_d, lay["qs"], lay["ks"], lay["vs"],
                              self.gran, **kw)

    def launches_per_step(self, fused=True):
        # one launch per fused layer, else the cache write and the decode kernel (the
        # split-counter reset is a memset node)
        return sum(1 if (fused and fz) else 2 for fz in self.fusable)

    def step_bytes(self):
        return sum(x["decode"] + x["write"] for x in self.bytes)


def _graph(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # eager warm-up on the capture stream (sets kernel attributes)
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def _time_graph(g, stream, steps, warmup, barrier):
    import torch
    with torch.cuda.stream(stream):      # CUDAGraph.replay launches on the current stream
        for _ in range(warmup):
            g.replay()
    stream.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1) / steps


def _step_distribution(g, stream, steps):
    """Per-replay times of a graph (an event pair around every replay, after the timed
    run): p10 / p50 / p90 in ms.  The events between replays add a little to each step,
    so these are for the spread; the headline uses the one event pair of _time_graph."""
    import numpy as np
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            g.replay()
            ev[i + 1].record(stream)
    ev[-1].synchronize()
    t = np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(steps)])
    p10, p50, p90 = np.percentile(t, [10, 50, 90])
    return {"steps": steps, "p10_ms": float(p10), "p50_ms": float(p50), "p90_ms": float(p90)}


def _time_replays(g, stream, n, flush=None):
    """Each of n replays of a graph timed alone by an event pair on the launching stream;
    ``flush`` (a buffer larger than the 129 MB L2) is overwritten before every replay,
    outside the pair, so that no replay finds the previous one's data in L2.  Returns
    the per-replay times in ms."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            if flush is not None:
                flush.zero_()
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def _pcts(ts):
    import numpy as np
    p10, p50, p90 = np.percentile(np.asarray(ts), [10, 50, 90])
    return {"p10": float(p10) * 1e3, "p50": float(p50) * 1e3, "p90": float(p90) * 1e3}


def _layer_kernels(f, st):
    """Which decode kernel each layer of a DecodeState runs, counted."""
    w = st.w
    names = {}
    for l, bf in enumerate(st.bf16):
        if not bf and f.fkv_decode_block_n(w.head_dim) > 0:
            k = f"decode_tc_kernel<{w.head_dim},{w.group}> (current-token write fused)"
        else:
            k = f"decode_split_kernel<{w.head_dim},{'bf16' if bf else 'e5m2'},{w.group}> (current-token write fused)"
        names[k] = names.get(k, 0) + 1
    return {k: f"{v} of {w.num_layers} layers" for k, v in names.items()}


def per_config(f, device, replays, peak, workloads=(1, 3, 4)):
    """The other decode workloads, each as one step of all its layers (current-token cache
    write + decode per layer, as the headline step), with an e4m3 cache and with the same
    kernels on a bf16 cache: per-replay times with an L2 flush before each replay (the
    single-layer 4096-key workload reads 8.4 MB, which L2 would otherwise hold), the
    algorithmic bytes of the step, GB/s and the fraction of the measured HBM peak."""
    import torch
    import synth
    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    out = {}
    for wid in workloads:
        w = synth.WORKLOADS[wid]
        entry = {"workload": w.name}
        for variant, kw in (("fp8", {}), ("bf16", {"all_bf16": True})):
            st = DecodeState(f, w, device, **kw)
            g = _graph(st.step, stream)
            _time_replays(g, stream, 3, flush)
            ts = _time_replays(g, stream, replays, flush)
            us = _pcts(ts)
            nbytes = st.step_bytes()
            gbs = nbytes / (us["p50"] * 1e-6) / 1e9
            entry[variant] = {"us_per_step": us, "replays": replays, "algorithmic_bytes": nbytes, "GBps": gbs,
                              "frac": gbs / peak, "kernels": _layer_kernels(f, st),
                              "launches_per_step": st.launches_per_step()}
            del g, st
            torch.cuda.empty_cache()
        entry["fp8_over_bf16_step_time"] = entry["fp8"]["us_per_step"]["p50"] / entry["bf16"]["us_per_step"]["p50"]
        out[str(wid)] = entry
    return out


def _fp8_dense_peak():
    """FP8 dense tensor peak: the measured bf16 GEMM peak times the nominal fp8/bf16 ratio 2."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return 2.0 * float(json.load(fh)["bf16_tflops"]), "measured bf16_tflops x 2 (nominal fp8/bf16)"
    return 2.0 * 1900.0, "fallback 1.9 PFLOP/s bf16 x 2"


def time_cache_write(f, device, peak, replays=20):
    """kv_quant_cache at fill size: the 131,072-token context of the needle workload (8 KV
    heads, head_dim 128, per-tensor scales) written into a shuffled e4m3 pool, timed per
    call with CUDA events, L2 flushed between calls.  Algorithmic bytes: the bf16 K and V
    read, the e4m3 codes written, the int64 slots read."""
    import numpy as np
    import torch
    import synth
    w = synth.WORKLOADS[4]
    ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
    table, nb = synth.block_table(ctx, seed=w.seed)
    data = synth.decode_layer(w, 0, ctx, device=device)
    cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim, device=device)
    slots = torch.from_numpy(synth.slot_mapping(table, ctx)).to(device)
    n = int(slots.numel())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    call = lambda: f.kv_quant_cache(data.k, data.v, slots, cache, data.k_scale, data.v_scale, f.SCALE_PER_TENSOR)
    for _ in range(3):
        call()
    ts = []
    for _ in range(replays):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    pc = _pcts(ts)
    by = n * w.num_kv_heads * w.head_dim * 2 * (2 + 1) + n * 8
    gbs = by / (pc["p50"] * 1e-6) / 1e9
    del data, cache, slots, flush
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}-fill", "kernel": "kv_quant_cache_kernel", "tokens": n,
            "us_p10_p50_p90": [pc["p10"], pc["p50"], pc["p90"]], "algorithmic_bytes": by,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak}}


def time_prefill(f, workload_id, device, iters, warmup, promote_every=(1,)):
    """Time fp8_prefill_attn on a prefill workload: the head_dim-256 causal batch (5) or the
    4096-query chunk over the 131072-key cache (4).  Algorithmic FLOPs = 4 * D * unmasked
    (query, key) pairs per head."""
    import numpy as np
    import torch
    import synth
    if workload_id == 5:
        w = synth.WORKLOADS[5]
        data = synth.prefill_data(w, device=device)
        ctx = np.full(w.batch, w.seq_len, np.int32)
        table, nb = synth.block_table(ctx, seed=w.seed)
        cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim, device=device)
        f.kv_quant_cache(data.k, data.v, torch.from_numpy(synth.slot_mapping(table, ctx)).to(device), cache,
                         data.k_scale, data.v_scale, f.SCALE_PER_HEAD)
        cu = torch.from_numpy(np.arange(w.batch + 1, dtype=np.int32) * w.seq_len).to(device)
        q, qs, ks, vs, L, gran = data.q, data.q_scale, data.k_scale, data.v_scale, w.seq_len, f.SCALE_PER_HEAD
        flops = 4 * w.head_dim * w.num_q_heads * w.batch * (w.seq_len * (w.seq_len + 1) // 2)
        name = w.name
        del data.k, data.v
    else:
        w = synth.WORKLOADS[4]
        ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
        table, nb = synth.block_table(ctx, seed=w.seed)
        data = synth.decode_layer(w, 0, ctx, device=device)
        cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim, device=device)
        f.kv_quant_cache(data.k, data.v, torch.from_numpy(synth.slot_mapping(table, ctx)).to(device), cache,
                         data.k_scale, data.v_scale, f.SCALE_PER_TENSOR)
        del data.k, data.v
        q = synth.prefill_query(w, 0, device=device)
        L = w.prefill_chunk
        cu = torch.tensor([0, L], dtype=torch.int32, device=device)
        qs, ks, vs, gran = data.q_scale, data.k_scale, data.v_scale, f.SCALE_PER_TENSOR
        T = int(ctx[0])
        flops = 4 * w.head_dim * w.num_q_heads * (L * (T - L) + L * (L + 1) // 2)
        name = w.name + f"-prefill{L}"
    tbl = torch.from_numpy(table).to(device)
    cx = torch.from_numpy(ctx).to(device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(device)

    res = []
    peak, kind = _fp8_dense_peak()
    for pe in promote_every:
        def call():
            f.fp8_prefill_attn(q, cu, L, cache, tbl, cx, qs, ks, vs, gran, out=out, stream=stream, promote_every=pe)

        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            call()
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / iters
        achieved = flops / (ms * 1e-3) / 1e12
        res.append({"workload": name, "promote_every": pe, "ms": ms, "flops": flops, "iters": iters,
                    "roofline": {"bound": "tensor", "kernel": "prefill_kernel", "achieved": achieved, "peak": peak,
                                 "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": kind}})
    return res


def linear_fit(xs, ys):
    """Least-squares line y = slope * x + intercept (the blog's ITL fit)."""
    n = len(xs)
    mx = sum(xs) / n
    my = sum(ys) / n
    sxx = sum((x - mx) ** 2 for x in xs)
    sxy = sum((x - mx) * (y - my) for x, y in zip(xs, ys))
    slope = sxy / sxx
    return slope, my - slope * mx


def break_even(slope_a, icpt_a, slope_b, icpt_b):
    """Context length where line a (e.g. FP8) drops below line b (e.g. BF16); None if it never does."""
    if slope_b <= slope_a:
        return None
    return (icpt_a - icpt_b) / (slope_b - slope_a)


def dist_barrier(dist, world):
    if world > 1:
        dist.barrier()


def dist_max(dist, world, x, device):
    """Maximum of a float over the ranks (all-reduce MAX)."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


SWEEP_T = (256, 1024, 2048, 4096, 8192, 16384, 32768, 65536, 125000)


ITL_SHORT_T = (1024, 4096, 16384, 65536, 125000)
TTFT_SHORT_L = (2048, 8192, 16384, 32768, 65536, 125000)


def itl_sweep(f, device, steps, warmup, lengths=SWEEP_T, shapes=("llama8b", "gptoss20b-hybrid")):
    """The ITL-slope proxy: per-step decode time of all layers at batch 1 versus the cached
    context T, for an e4m3 cache and for a bf16 cache, with least-squares lines (the blog's
    ITL = slope * input_len + intercept) and the break-even context.  Shapes: the
    Llama-3.1-8B-shaped stack (32 layers, 32/8 heads, head_dim 128) and the gpt-oss-20b-shaped
    hybrid stack (24 layers, window-128 layers every other layer), the latter with and
    without the sliding-window layers kept bf16."""
    import dataclasses
    import torch
    import synth
    out = {}
    all_shapes = {"llama8b": (synth.WORKLOADS[2], [("fp8", {}), ("bf16", {"all_bf16": True})]),
                  "gptoss20b-hybrid": (synth.WORKLOADS[3], [("fp8-skip-sw", {}), ("fp8", {"no_skip": True}),
                                                            ("bf16", {"all_bf16": True})])}
    stream = torch.cuda.Stream(device)
    # short contexts fit in L2 (32 layers x 1024 keys of e4m3 = 67 MB): flush before each replay
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    for name in shapes:
        base, variants = all_shapes[name]
        res = {v: [] for v, _ in variants}
        for T in lengths:
            w = dataclasses.replace(base, batch=1, ctx_lo=T, ctx_hi=T, name=f"{base.name}-b1-t{T}")
            for v, kw in variants:
                st = DecodeState(f, w, device, **kw)
                g = _graph(st.step, stream)
                _time_replays(g, stream, warmup, flush)
                res[v].append(_pcts(_time_replays(g, stream, steps, flush))["p50"])
                del g, st
                torch.cuda.empty_cache()
        entry = {"T": list(lengths), "us_per_step": res, "timing": "median of per-replay times, L2 flushed"}
        fits = {v: linear_fit(list(lengths), ys) for v, ys in res.items()}
        entry["slope_us_per_1k_tokens"] = {v: fi[0] * 1e3 for v, fi in fits.items()}
        entry["intercept_us"] = {v: fi[1] for v, fi in fits.items()}
        ref = fits["bf16"]
        entry["slope_ratio_vs_bf16"] = {v: fi[0] / ref[0] for v, fi in fits.items() if v != "bf16"}
        entry["break_even_tokens"] = {v: break_even(fi[0], fi[1], ref[0], ref[1])
                                      for v, fi in fits.items() if v != "bf16"}
        out[name] = entry
    return out


def quadratic_fit(xs, ys):
    """Least-squares TTFT = a * L^2 + b * L + c (the blog's quadratic TTFT model).  The
    lengths are scaled by 1/1000 for the solve, so the normal matrix stays well conditioned."""
    import numpy as np
    x = np.asarray(xs, dtype=np.float64) / 1000.0
    A = np.stack([x * x, x, np.ones_like(x)], axis=1)
    a, b, c = np.linalg.lstsq(A, np.asarray(ys, dtype=np.float64), rcond=None)[0]
    return float(a) / 1e6, float(b) / 1e3, float(c)


def ttft_sweep(f, device, steps, warmup, lengths=SWEEP_T, shape_names=("llama8b", "hd256")):
    """The TTFT proxy: one layer's prefill of a single prompt of L tokens (cache write of
    its K/V + causal attention over it) versus L, fitted with TTFT = a L^2 + b L + c, for
    an e4m3 cache (two-level accumulation, and without promotion) and a bf16 cache.
    Shapes: Llama-3.1-8B-shaped (32/8 heads, head_dim 128) and the head_dim-256 shape
    (8/1 heads) whose FP8/BF16 ratio of the quadratic coefficient the blog reports as ~1.6
    with two-level accumulation on H100.  The prompts of all lengths are prefixes of one
    seeded draw.  No L2 flush: the step is tensor-bound and re-reads its own inputs."""
    import dataclasses
    import numpy as np
    import torch
    import synth
    Lmax = max(lengths)
    shapes = {
        "llama8b": synth.PrefillWorkload("llama8b-prefill-h32x8-d128", 1, Lmax, 32, 8, 128, seed=1),
        "hd256": dataclasses.replace(synth.WORKLOADS[5], batch=1, seq_len=Lmax, name="prefill-h8x1-d256"),
    }
    shapes = {k: v for k, v in shapes.items() if k in shape_names}
    variants = [("fp8", 1, False), ("fp8-no-promote", 0, False), ("bf16", 1, True)]
    stream = torch.cuda.Stream(device)
    out = {}
    for name, w in shapes.items():
        data = synth.prefill_data(w, device=device)
        ctx_max = np.array([Lmax], np.int32)
        table, nb = synth.block_table(ctx_max, seed=w.seed)
        slots = torch.from_numpy(synth.slot_mapping(table, ctx_max)).to(device)
        tbl = torch.from_numpy(table).to(device)
        res = {v: [] for v, _, _ in variants}
        for v, pe, bf in variants:
            cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim, bf16=bf, device=device)
            mask = [1] if bf else None
            qs, ks, vs = (None, None, None) if bf else (data.q_scale, data.k_scale, data.v_scale)
            outb = torch.empty_like(data.q)
            for L in lengths:
                cu = torch.tensor([0, L], dtype=torch.int32, device=device)
                cx = torch.tensor([L], dtype=torch.int32, device=device)

                def step():
                    f.kv_quant_cache(data.k[:L], data.v[:L], slots[:L], cache, ks, vs, f.SCALE_PER_HEAD, layer=0,
                                     skip_layer_mask=mask, stream=stream)
                    f.fp8_prefill_attn(data.q[:L], cu, L, cache, tbl, cx, qs, ks, vs, f.SCALE_PER_HEAD, causal=True,
                                       promote_every=pe, layer=0, skip_layer_mask=mask, out=outb[:L], stream=stream)

                g = _graph(step, stream)
                res[v].append(_time_graph(g, stream, steps, warmup, lambda: None))
                del g
            del cache, outb
            torch.cuda.empty_cache()
        fits = {v: quadratic_fit(lengths, ys) for v, ys in res.items()}
        flops = [4 * w.head_dim * w.num_q_heads * (L * (L + 1) // 2) for L in lengths]
        out[name] = {
            "L": list(lengths), "ms": res,
            "attn_tflops": {v: [fl / (ms * 1e-3) / 1e12 for fl, ms in zip(flops, ys)] for v, ys in res.items()},
            "fit_ms": {v: {"a_per_tok2": a, "b_per_tok": b, "c": c} for v, (a, b, c) in fits.items()},
            "a_ratio_vs_bf16": {v: fits[v][0] / fits["bf16"][0] for v in fits if v != "bf16"},
            "ttft_ratio_vs_bf16_at_max": {v: res[v][-1] / res["bf16"][-1] for v in res if v != "bf16"},
        }
        del data
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(workload_id: int, keys: int, heads: int):
    """Time the oracle on one sequence of layer 0: its cache write (quantise K/V) and its
    decode attention for ``heads`` query heads (heads / G KV heads) over ``keys`` cached
    keys, with the workload's scale recipe (1.0, or amax/448 per head).  Returns
    (seconds, algorithmic bytes of that sample: the e4m3 K/V it reads)."""
    import numpy as np
    import synth
    from oracle import attention
    w = synth.WORKLOADS[workload_id]
    G = w.group
    nkv = max(1, heads // G)
    q = synth.randn_bf16((heads, w.head_dim), w.seed, 0, "q")
    k = synth.randn_bf16((keys, nkv, w.head_dim), w.seed, 0, "k")
    v = synth.randn_bf16((keys, nkv, w.head_dim), w.seed, 0, "v")
    if w.scale_mode == "amax":
        qs, ks, vs = (synth.amax_scales(x, 1).numpy() for x in (q, k, v))
    else:
        qs = ks = vs = np.ones(1, np.float32)
    qf, kf, vf = synth.bf16_to_f64(q), synth.bf16_to_f64(k), synth.bf16_to_f64(v)
    t0 = time.perf_counter()
    attention.decode_attention_contiguous(qf, kf, vf, qs, ks, vs, fp8=True)
    dt = time.perf_counter() - t0
    return dt, 2 * nkv * w.head_dim * keys


def oracle_sample_shape(workload_id: int):
    """The bounded sample both CPU legs time, one per step: layer 0, sequence 0 of the
    workload (its whole context), KV head 0 and its G query heads.  Returns (keys, heads,
    description)."""
    import synth
    w = synth.WORKLOADS[workload_id]
    ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
    keys = int(ctx[0])
    return keys, w.group, (f"layer 0, sequence 0 of {w.batch}: {keys} cached keys of KV head 0 x its {w.group} "
                           f"query heads: e4m3 cache quantisation + decode attention in float64 NumPy")


def _cpu_baseline_subprocess(workload_id: int, repeats: int):
    """The oracle sample timed ``repeats`` times in a fresh single-threaded process (no
    CUDA context).  Returns (seconds, bytes) summed over the repeats, or None."""
    keys, heads, _ = oracle_sample_shape(workload_id)
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    code = (f"import bench, json; r = [bench.oracle_sample({workload_id}, {keys}, {heads}) for _ in range({repeats})]; "
            f"print(json.dumps({{'s': sum(x[0] for x in r), 'bytes': sum(x[1] for x in r)}}))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return None
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["s"], d["bytes"]


def _host_cores():
    return {"host_cpu_count": os.cpu_count(), "blas_threads": 1,
            "threads_note": "the oracle runs single-threaded (OPENBLAS/OMP/MKL_NUM_THREADS=1)"}


def workload_config(w, ctx, world, step_bytes=None):
    """The ``config`` object of both arms' JSON lines for a decode workload."""
    cfg = {"workload": w.name, "layers": w.num_layers, "batch": w.batch, "q_heads": w.num_q_heads,
           "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "context": [int(x) for x in ctx], "block_size": 16,
           "kv_cache_dtype": "e4m3", "scales": "per-KV-head amax/448" if w.scale_mode == "amax" else "per-tensor 1.0",
           "l2": "no flush: each step reads {:.2f} GB (> 129 MB L2)".format(
               (step_bytes if step_bytes is not None else _step_bytes_host(w, ctx)) / 1e9),
           "graph": "one CUDA graph per step", "parallelism": f"replicas x{world}"}
    return cfg


def _step_bytes_host(w, ctx):
    bf = [bool(x) for x in w.skip_mask()]
    return sum(x["decode"] + x["write"] for x in decode_bytes(w, ctx, bf))


# ----------------------------------------------------------------------------- arms

def run_reference(args):
    """The reference arm: the CPU oracle as it stands, one bounded sample per step (the
    same sample as the benchmark line's cpu_baseline)."""
    import synth
    rank, world, _ = _env_rank()
    if rank != 0:
        return 0
    w = synth.WORKLOADS[args.workload]
    keys, heads, sample = oracle_sample_shape(args.workload)
    for _ in range(args.warmup):
        oracle_sample(args.workload, keys, heads)
    tot_s, tot_b = 0.0, 0
    for _ in range(args.steps):
        s_, b = oracle_sample(args.workload, keys, heads)
        tot_s += s_
        tot_b += b
    value = tot_b / tot_s / 1e9
    ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, ctx, args.gpus),
        "cpu_baseline": dict({"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                              "sample": sample + " (one sample per step)"}, **_host_cores()),
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    import fp8_kv_cache_quant_gb300 as f
    import synth

    rank, world, local = _env_rank()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        dist_barrier(dist, world)

    def max_over_ranks(x):
        return dist_max(dist, world, x, device)

    f.load_library()
    if args.sweep or args.ttft:
        if args.sweep:
            res = itl_sweep(f, device, steps=max(3, min(args.steps, 50)), warmup=args.warmup)
            if rank == 0:
                print(json.dumps({"sweep": "ITL-slope proxy (decode step time vs cached context, batch 1)",
                                  "unit": "us", "results": res}), flush=True)
        if args.ttft:
            res = ttft_sweep(f, device, steps=max(2, min(args.steps, 5)), warmup=min(args.warmup, 3))
            if rank == 0:
                print(json.dumps({"sweep": "TTFT proxy (one layer's prompt prefill: cache write + causal "
                                  "attention, vs prompt length)", "unit": "ms", "results": res}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return 0
    w = synth.WORKLOADS[args.workload]
    stream = torch.cuda.Stream(device)

    fp8 = DecodeState(f, w, device)
    g_fp8 = _graph(fp8.step, stream)
    g_dec = _graph(lambda: fp8.step(decode_only=True), stream)
    # the same step with the cache write as its own launch, like for like with the bf16 step
    g_sep = _graph(lambda: fp8.step(fused=False), stream) if not args.no_bf16 else None

    # end to end: pinned host inputs -> device, the step, outputs -> pinned host
    host_in = [t.to("cpu").pin_memory() for t in (fp8.q_all, fp8.k_all, fp8.v_all)]
    host_out = torch.empty_like(fp8.out_all, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        for h, d in zip(host_in, (fp8.q_all, fp8.k_all, fp8.v_all)):
            d.copy_(h, non_blocking=True)
        fp8.step()
        host_out.copy_(fp8.out_all, non_blocking=True)

    g_e2e = _graph(e2e_step, stream)

    clocks = ClockSampler(local)
    clocks.start()
    ms_fp8 = max_over_ranks(_time_graph(g_fp8, stream, args.steps, args.warmup, barrier))
    ms_dec = max_over_ranks(_time_graph(g_dec, stream, args.steps, args.warmup, barrier))
    ms_e2e = max_over_ranks(_time_graph(g_e2e, stream, args.steps, args.warmup, barrier))
    ms_sep = max_over_ranks(_time_graph(g_sep, stream, args.steps, args.warmup, barrier)) if g_sep else None
    spread = _step_distribution(g_fp8, stream, args.steps)
    clocks.stop()

    step_bytes = fp8.step_bytes()
    value = world * step_bytes / (ms_fp8 * 1e-3) / 1e9
    e2e_value = world * step_bytes / (ms_e2e * 1e-3) / 1e9
    dec_bytes = sum(x["decode"] for x in fp8.bytes) / w.num_layers
    dec_launch_ms = ms_dec / w.num_layers
    peak, peak_kind = _peaks()
    achieved = dec_bytes / (dec_launch_ms * 1e-3) / 1e9
    # the decode kernel this workload's e4m3 layers run: tensor cores (head_dim 128 / 256) or CUDA cores
    if f.fkv_decode_block_n(w.head_dim) > 0:
        dec_kernel = "decode_tc_kernel (fp8_decode_attn on tcgen05, merge fused)"
        traffic = _traffic_record("decode_tc.cu", "decode_tc_llama8b_decode.txt")
    else:
        dec_kernel = "decode_split_kernel (fp8_decode_attn on CUDA cores, merge fused)"
        traffic = _traffic_record("decode_attn.cu", "decode_attn_llama8b_decode.txt")

    # the same step with a bf16 cache (all layers), for the FP8-vs-BF16 per-token cost
    bf16_info = None
    if not args.no_bf16:
        bf = DecodeState(f, w, device, all_bf16=True)
        g_bf = _graph(bf.step, stream)
        ms_bf = max_over_ranks(_time_graph(g_bf, stream, args.steps, args.warmup, barrier))
        bf_bytes = bf.step_bytes()
        kv_fp8 = sum(x["kv"] for x in fp8.bytes)
        kv_bf = sum(x["kv"] for x in bf.bytes)
        g_bf_sep = _graph(lambda: bf.step(fused=False), stream)
        ms_bf_sep = max_over_ranks(_time_graph(g_bf_sep, stream, args.steps, args.warmup, barrier))
        bf16_info = {"ms_per_step": ms_bf, "GBps": bf_bytes / (ms_bf * 1e-3) / 1e9,
                     # both steps fused (one launch per layer: cache write + decode)
                     "fp8_over_bf16_step_time": ms_fp8 / ms_bf,
                     # both steps with the cache write as its own launch
                     "fp8_over_bf16_step_time_unfused": ms_sep / ms_bf_sep,
                     "fp8_unfused_ms_per_step": ms_sep, "bf16_unfused_ms_per_step": ms_bf_sep,
                     "kv_bytes_fp8": kv_fp8, "kv_bytes_bf16": kv_bf}
        del g_bf_sep

    fp8_ctx, fp8_launches = fp8.ctx, fp8.launches_per_step()
    del fp8, g_fp8, g_dec, g_e2e, g_sep
    if not args.no_bf16:
        del bf, g_bf
    torch.cuda.empty_cache()
    clocks_x = ClockSampler(local)   # clocks of the remaining measurements
    clocks_x.start()
    prefill = None
    if not args.no_prefill:
        torch.cuda.synchronize()
        prefill = (time_prefill(f, 5, device, iters=min(args.steps, 10), warmup=3, promote_every=(1, 4, 0)) +
                   time_prefill(f, 4, device, iters=min(args.steps, 10), warmup=3, promote_every=(1, 4, 0)))
        torch.cuda.synchronize()

    cache_write = None
    if not args.no_prefill:
        cache_write = time_cache_write(f, device, peak)

    # the other decode workloads, the ITL-slope proxy and the TTFT fit (short forms of
    # --sweep / --ttft), each on this GPU in the same run
    others = None
    if not args.no_per_config:
        others = per_config(f, device, replays=max(20, min(args.steps, 100)), peak=peak)
    itl = None
    if not args.no_itl:
        itl = itl_sweep(f, device, steps=max(10, min(args.steps, 30)), warmup=3, lengths=ITL_SHORT_T,
                        shapes=("llama8b",))
    ttft = None
    if not args.no_ttft:
        ttft = ttft_sweep(f, device, steps=3, warmup=2, lengths=TTFT_SHORT_L)
    clocks_x.stop()

    cpu = None
    if rank == 0 and not args.no_cpu:
        repeats = 20
        r = _cpu_baseline_subprocess(args.workload, repeats)
        if r is not None:
            s, b = r
            _, _, sample = oracle_sample_shape(args.workload)
            cpu = dict({"value": b / s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                        "sample": f"{sample}, timed {repeats} times ({s:.1f} s)"}, **_host_cores())

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_fp8, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, fp8_ctx, world),
            "us_per_step": ms_fp8 * 1e3,
            "step_ms_spread": spread,
            "pct_of_hbm_peak": value / peak,
            "roofline": {"bound": "hbm", "kernel": dec_kernel,
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": f"{peak_kind} hbm_gbs", "traffic": traffic,
                         "algorithmic_bytes_per_launch": dec_bytes, "launch_ms": dec_launch_ms},
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": ms_e2e},
            "gpu_launches": fp8_launches * args.steps,
            "clocks": clocks.summary(),
            "clocks_other_measurements": clocks_x.summary(),
            "bf16": bf16_info,
            "prefill": prefill,
            "cache_write": cache_write,
            "per_config": others,
            "itl_slope": itl,
            "ttft_fit": ttft,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other decode workloads")
    ap.add_argument("--no-itl", action="store_true", help="skip the short ITL-slope sweep")
    ap.add_argument("--no-ttft", action="store_true", help="skip the short TTFT fit")
    ap.add_argument("--sweep", action="store_true", help="ITL-slope sweep instead of the benchmark line")
    ap.add_argument("--ttft", action="store_true", help="TTFT quadratic-fit sweep instead of the benchmark line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
