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


# The prefill rounds P per tile of this many keys (fp8kv.h: fkv_prefill_block_n); the
# tests pass it to the oracle and check that the library agrees.
PREFILL_BLOCK_N = 128


def decode_block_n(head_dim):
    """Keys per tile over which the tensor-core decode of e4m3 layers rounds P, restated
    from include/fp8kv.h (fkv_decode_block_n): 256 at head_dim 64, else 128."""
    return 256 if head_dim == 64 else 128


def decode_split_blocks(max_blocks, window, num_splits, head_dim=128):
    """Blocks per context split of fp8_decode_attn for a requested split count, restated
    from the rule include/fp8kv.h documents: n = max_blocks, or with a window W at most
    ceil(W / 16) + 1 blocks; ceil(n / num_splits), at most 256 and at least
    ceil(n / 1024), rounded up to a multiple of u, the blocks of one decode tile."""
    assert num_splits > 0
    u = decode_block_n(head_dim) // 16
    n = max_blocks if window <= 0 else min(max_blocks, -(-window // 16) + 1)
    bps = min(-(-n // num_splits), 256)
    bps = max(bps, -(-n // 1024), 1)
    return -(-bps // u) * u


def auto_split_blocks(batch, num_kv_heads, max_blocks, window, num_sms, head_dim=128):
    """The automatic plan (num_splits 0) restated from include/fp8kv.h: the multiple of u
    (the blocks of one decode tile) up to 256 minimising waves * blocks per split, waves
    counted on 3 resident CTAs per SM, ties to the larger count."""
    u = decode_block_n(head_dim) // 16
    n = max_blocks if window <= 0 else min(max_blocks, -(-window // 16) + 1)
    units, slots = max(batch, 1) * num_kv_heads, 3 * num_sms
    best = None
    for c in range(u, 257, u):
        ctas = units * -(-n // c)
        cost = -(-ctas // slots) * min(c, n)
        if best is None or cost < best[1] or (cost == best[1] and c > best[0]):
            best = (c, cost)
    bps = max(best[0], -(-n // 1024))
    return -(-bps // u) * u


def assert_within_p_bound(gpu, exact, bound, what=""):
    """The tensor-core decode against the plain softmax definition (P exact, reading R9 of
    the exact result): its output may differ by the rounding of P to e4m3, at most the
    oracle's p_rounding_bound B per element, plus the kernel's own arithmetic — the
    bf16 rounding of the output (2^-9 relative) and FP32 scores and sums (relative errors
    below 1e-4 of the weights) — covered by the factor 1 + 2^-6 on B and 2^-8 |o|.
    Returns (rel-L2 distance, largest |gpu - exact| / B)."""
    gpu = np.asarray(gpu, np.float64)
    exact = np.asarray(exact, np.float64)
    bound = np.asarray(bound, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - exact)
    tol = bound * (1 + 2.0 ** -6) + 2.0 ** -8 * np.abs(exact)
    worst = int(np.argmax(err - tol))
    assert np.all(err <= tol), (f"{what}: |gpu - exact| {err.flat[worst]:.3e} above {tol.flat[worst]:.3e} "
                                f"(bound {bound.flat[worst]:.3e}) at {np.unravel_index(worst, err.shape)}")
    ratio = float(np.max(err / np.where(bound > 0, bound, np.inf))) if err.size else 0.0
    return rel_l2(gpu, exact), ratio
