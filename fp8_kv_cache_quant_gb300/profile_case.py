"""Run one workload layer's kernels a few times, eagerly, for ncu captures.

    python -m fp8_kv_cache_quant_gb300.profile_case --workload 2 --layer 0 --iters 3 [--bf16]
    python -m fp8_kv_cache_quant_gb300.profile_case --workload 4 --fill --iters 3

Builds one layer of a decode workload (seeded synthetic inputs, pool filled by
kv_quant_cache) and launches fp8_decode_attn ``iters`` times.  The layer's cache is
larger than L2 for the Llama-shaped workload (335 MB), so DRAM counters are meaningful,
and the device holds about 1 GB.  It prints nothing but a final line; it is not a
benchmark.
"""
from __future__ import annotations

import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def main():
    import numpy as np
    import torch

    import fp8_kv_cache_quant_gb300 as f
    import synth

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--layer", type=int, default=0)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--bf16", action="store_true", help="bf16 pool (the skip-layer path) instead of e4m3")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--step", action="store_true",
                    help="decode through fp8_decode_step (the current token's cache write in the same launch)")
    ap.add_argument("--prefill", action="store_true",
                    help="run fp8_prefill_attn on the head_dim-256 prefill shape instead (batch 1)")
    ap.add_argument("--llama", action="store_true",
                    help="with --prefill: the Llama-3.1-8B head shape (32/8 heads, head_dim 128)")
    ap.add_argument("--seq", type=int, default=8192, help="prefill sequence length")
    ap.add_argument("--fill", action="store_true",
                    help="run kv_quant_cache over the workload's whole context (one layer's fill) instead")
    a = ap.parse_args()
    if a.prefill:
        return run_prefill(a)
    if a.fill:
        return run_fill(a)
    w = synth.WORKLOADS[a.workload]
    dev = torch.device("cuda:0")
    ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
    table, nb = synth.block_table(ctx, seed=w.seed)
    data = synth.decode_layer(w, a.layer, ctx, device=dev)
    mask = np.array([1 if a.bf16 else 0], np.uint8)
    gran = f.SCALE_PER_HEAD if w.scale_mode == "amax" else f.SCALE_PER_TENSOR
    cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim, bf16=a.bf16, device=dev)
    slots = torch.from_numpy(synth.slot_mapping(table, ctx)).to(dev)
    f.kv_quant_cache(data.k, data.v, slots, cache, data.k_scale, data.v_scale, gran, layer=0, skip_layer_mask=mask)
    last = torch.from_numpy(np.cumsum(ctx) - 1).to(dev)
    k_new, v_new = data.k[last].contiguous(), data.v[last].contiguous()  # each sequence's current token
    del data.k, data.v
    table_d = torch.from_numpy(table).to(dev)
    ctx_d = torch.from_numpy(ctx).to(dev)
    out = torch.empty_like(data.q)
    ws = f.decode_workspace(w.batch, w.num_q_heads, cache, table.shape[1], w.layer_window(a.layer), a.splits, dev)
    for _ in range(a.iters):
        if a.step:
            f.fp8_decode_step(k_new, v_new, data.q, cache, table_d, ctx_d, data.q_scale, data.k_scale, data.v_scale,
                              gran, window=w.layer_window(a.layer), layer=0, skip_layer_mask=mask, out=out,
                              workspace=ws, num_splits=a.splits)
        else:
            f.fp8_decode_attn(data.q, cache, table_d, ctx_d, data.q_scale, data.k_scale, data.v_scale, gran,
                              window=w.layer_window(a.layer), layer=0, skip_layer_mask=mask, out=out, workspace=ws,
                              num_splits=a.splits)
    torch.cuda.synchronize()
    print("profile_case done", w.name, "layer", a.layer, "bf16" if a.bf16 else "e4m3")


def run_fill(a):
    import torch

    import fp8_kv_cache_quant_gb300 as f
    import synth

    w = synth.WORKLOADS[a.workload]
    dev = torch.device("cuda:0")
    ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
    table, nb = synth.block_table(ctx, seed=w.seed)
    data = synth.decode_layer(w, a.layer, ctx, device=dev)
    gran = f.SCALE_PER_HEAD if w.scale_mode == "amax" else f.SCALE_PER_TENSOR
    cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim, device=dev)
    slots = torch.from_numpy(synth.slot_mapping(table, ctx)).to(dev)
    for _ in range(a.iters):
        f.kv_quant_cache(data.k, data.v, slots, cache, data.k_scale, data.v_scale, gran)
    torch.cuda.synchronize()
    print("profile_case done fill", w.name, int(slots.numel()), "tokens")


def run_prefill(a):
    import numpy as np
    import torch

    import fp8_kv_cache_quant_gb300 as f
    import synth

    w = synth.WORKLOADS[5]
    if a.llama:
        w = synth.PrefillWorkload("llama8b-prefill-h32x8-d128", 1, a.seq, 32, 8, 128, seed=1)
    dev = torch.device("cuda:0")
    data = synth.prefill_data(w, device=dev, seq_len=a.seq, batch=1)
    ctx = np.array([a.seq], np.int32)
    table, nb = synth.block_table(ctx, seed=w.seed)
    cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim, device=dev)
    f.kv_quant_cache(data.k, data.v, torch.from_numpy(synth.slot_mapping(table, ctx)).to(dev), cache, data.k_scale,
                     data.v_scale, f.SCALE_PER_HEAD)
    cu = torch.tensor([0, a.seq], dtype=torch.int32, device=dev)
    tbl = torch.from_numpy(table).to(dev)
    cx = torch.from_numpy(ctx).to(dev)
    out = torch.empty_like(data.q)
    for _ in range(a.iters):
        f.fp8_prefill_attn(data.q, cu, a.seq, cache, tbl, cx, data.q_scale, data.k_scale, data.v_scale,
                           f.SCALE_PER_HEAD, out=out)
    torch.cuda.synchronize()
    print("profile_case done prefill", a.seq)


if __name__ == "__main__":
    main()
