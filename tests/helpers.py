"""Shared helpers of the GPU tests: build paged layers through the C ABI from the seeded
synthetic inputs, and compare against the oracle with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Tolerances of attention outputs against the oracle's float64 result (FP8-emulated):
# max-abs 2e-2 and relative L2 1e-2, as the problem statement fixes them.
MAX_ABS = 2e-2
REL_L2 = 1e-2


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


def assert_close(gpu, ref, max_abs=MAX_ABS, rl2=REL_L2, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    ma = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    r = rel_l2(gpu, ref)
    assert ma <= max_abs and r <= rl2, f"{what}: max_abs={ma:.3e} rel_l2={r:.3e}"
    return ma, r


def to_dev(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def build_layer(f, ctx, table, num_blocks, k, v, ks, vs, gran, bf16_layer, sentinel=None, kv_format=0):
    """Allocate one layer's pools and fill them with kv_quant_cache (all positions)."""
    H, D = k.shape[1], k.shape[2]
    cache = f.LayerCache.empty(num_blocks, H, D, bf16=bf16_layer, kv_format=kv_format)
    if sentinel is not None:
        cache.k_cache.view(torch.uint8).fill_(sentinel)
        cache.v_cache.view(torch.uint8).fill_(sentinel)
    slots = to_dev(synth.slot_mapping(table, ctx))
    f.kv_quant_cache(k.cuda().contiguous(), v.cuda().contiguous(), slots, cache, to_dev(ks), to_dev(vs), gran,
                     layer=0, skip_layer_mask=[1] if bf16_layer else None)
    return cache


def seq_slices(ctx):
    cu = np.concatenate([[0], np.cumsum(ctx)])
    return [(int(cu[b]), int(cu[b + 1])) for b in range(len(ctx))]


def oracle_pools(oracle_kvcache, ctx, table, num_blocks, k, v, ks, vs, bf16_layer, fmt="e4m3"):
    """The oracle's own pools, written by the oracle's cache write from the bf16 inputs."""
    H, D = k.shape[1], k.shape[2]
    if bf16_layer:
        kp = np.zeros((num_blocks, H, 16, D))
        vp = np.zeros((num_blocks, H, 16, D))
    else:
        kp = np.zeros((num_blocks, H, 16, D), np.uint8)
        vp = np.zeros((num_blocks, H, 16, D), np.uint8)
    slots = synth.slot_mapping(table, ctx)
    oracle_kvcache.cache_write(synth.bf16_to_f64(k), synth.bf16_to_f64(v), slots, kp, vp,
                               np.asarray(ks, np.float32), np.asarray(vs, np.float32), skip=bf16_layer, fmt=fmt)
    return kp, vp
