"""Paged KV-cache write and the KV memory formula (float64 / integer NumPy).

Cache write: the pages' ``reshape_and_cache_flash`` writes each new token's K and V
into the paged cache, quantised with either one scale or an array with one scale
per KV head (vLLM blog, section "Kernel 与 vLLM 改进", paragraph "Per-Head Scales").
Layers named by the skip-layer mask stay bf16 (same section, paragraph "跳过 Layer",
flag ``--kv-cache-dtype-skip-layers``).

Pool layout (the pages are silent; the reading taken): per layer
``[num_blocks][H_kv][block_size][D]``, one byte per element for e4m3 and two for
bf16; token position p of a sequence lives in physical slot
``block_table[p // bs] * bs + p % bs``; a negative slot means "padding, skip".
"""
from __future__ import annotations

import numpy as np

from . import e4m3, e5m2


def head_scale(scale, h: int) -> float:
    """Scale of head h from a [1] (per-tensor) or [H] (per-head) array."""
    s = np.asarray(scale, dtype=np.float32).reshape(-1)
    return float(s[0] if s.size == 1 else s[h])


def cache_write(k, v, slots, k_pool, v_pool, k_scale, v_scale, *, skip: bool, block_size: int = 16,
                fmt: str = "e4m3"):
    """Write tokens into the pools in place.

    k, v: float64 [n][H_kv][D] holding bf16 values (or, for ``skip``, uint16 bf16
    bit patterns may be passed instead).  k_pool / v_pool: uint8 codes
    ``[nb][H_kv][bs][D]`` (an FP8 layer, format ``fmt``: "e4m3" or "e5m2") or uint16
    bf16 bits (skip layer).  Every byte not addressed by a non-negative slot keeps its
    prior value.
    """
    codec = {"e4m3": e4m3, "e5m2": e5m2}[fmt]
    slots = np.asarray(slots, dtype=np.int64)
    n, H, D = np.shape(k)
    for t in range(n):
        s = int(slots[t])
        if s < 0:
            continue
        blk, off = s // block_size, s % block_size
        for h in range(H):
            if skip:
                k_pool[blk, h, off, :] = k[t, h]
                v_pool[blk, h, off, :] = v[t, h]
            else:
                k_pool[blk, h, off, :] = codec.quantize(k[t, h], head_scale(k_scale, h))
                v_pool[blk, h, off, :] = codec.quantize(v[t, h], head_scale(v_scale, h))
    return k_pool, v_pool


def clip_count(x, scale, limit: float = e4m3.E4M3_MAX) -> int:
    """Number of elements whose scaled value fl32(x * fl32(1/scale)) lies beyond the FP8
    range, |y| > limit (448 for e4m3, 57344 for e5m2), and is therefore clipped by the
    saturating encode — the clipping frequency the KV-cache quantisation explainer asks
    to watch when it can be observed ("本番投入前の比較" checklist).  NaN is not counted.
    ``x``: float64 [n][H][D] (bf16 values); ``scale``: one value or one per head (axis 1)."""
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(scale, dtype=np.float32).reshape(-1)
    inv = e4m3.reciprocal_f32(s if s.size == 1 else s.reshape(1, -1, 1))
    y = e4m3.fl32(x * inv)
    with np.errstate(invalid="ignore"):
        return int(np.count_nonzero(np.abs(y) > limit))


def kv_bytes_formula(num_layers, num_kv_heads, head_dim, tokens, batch, elem_bytes) -> int:
    """M_KV = 2 * L * H_KV * D * T * B * S (vLLM-independent explainer "KV Cache量子化とは？",
    section "weight量子化とは別の場所を小さくする", the KV memory formula)."""
    return 2 * num_layers * num_kv_heads * head_dim * tokens * batch * elem_bytes


def paged_kv_bytes(num_kv_heads, head_dim, context_lens, elem_bytes_per_layer, block_size=16) -> int:
    """The same formula with each sequence rounded up to whole blocks (the explainer's
    "block単位の余り"), summed over layers of possibly different element size."""
    blocks = sum((int(t) + block_size - 1) // block_size for t in context_lens)
    return sum(2 * num_kv_heads * head_dim * block_size * blocks * s for s in elem_bytes_per_layer)
