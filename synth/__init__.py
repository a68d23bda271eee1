"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only *draws* inputs: bf16 activations, paged block tables, context
lengths, slot mappings and the per-head scale arrays that both sides receive as
inputs.  It holds none of the quantisation or attention arithmetic; the CUDA
library and the CPU oracle each implement that on their own.

Workload shapes follow the pages' workloads (vLLM blog "FP8 KV-Cache and
Attention quantization in vLLM", section "性能 Benchmark": Llama-3.1-8B and
gpt-oss-20b decode, the 128k needle test, head_dim 256 prefill of gemma-4-E2B).
No dataset or trained weight is used; every tensor is drawn from a seeded
generator.

Recipe (stated once, used everywhere):
  * activations: float32 N(0,1) from ``torch.Generator`` seeded per
    (workload seed, layer, tensor kind), rounded to bf16 (round-to-nearest-even);
  * K outliers: ``k_outliers`` channels per (layer, KV head), chosen by the same
    seed, multiplied by 8 before the bf16 rounding;
  * context lengths: integers uniform in [ctx_lo, ctx_hi] from the seed;
  * block table: one seeded random permutation of all physical blocks, handed
    out to (sequence, logical block) in order; unused table entries are -1;
  * scales: either 1.0 (the pages' uncalibrated default) or amax/448 per
    (layer, head, K or V), amax taken over all tokens in float64 and rounded to
    float32 once;
  * the long-context needle: for KV head g the key at a seeded position equals
    4*sqrt(D)*q/||q|| of query head g*G (before bf16 rounding).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

BLOCK_SIZE = 16
E4M3_MAX = 448.0

# tensor-kind tags used to derive independent generator streams
_KIND = {"q": 1, "k": 2, "v": 3, "outlier": 4, "ctx": 5, "table": 6, "needle": 7, "qp": 8}


def _gen(seed: int, layer: int, kind: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + layer * 7919 + _KIND[kind] * 104_729) % (2**63 - 1))
    return g


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One paged decode workload (all layers share the block table)."""

    name: str
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx_lo: int
    ctx_hi: int
    seed: int
    scale_mode: str = "unit"          # "unit" -> 1.0 ; "amax" -> amax/448 per head
    k_outliers: int = 0               # channels scaled x8 per (layer, KV head)
    window: int = 0                   # sliding window of the SW layers
    sw_layers: tuple = ()             # indices of sliding-window layers
    skip_sw: bool = False             # SW layers kept bf16 by the skip-layer mask
    needle: bool = False              # plant the long-context needle (R15)
    prefill_chunk: int = 0            # length of the FP8 prefill chunk over the same cache

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def layer_window(self, layer: int) -> int:
        return self.window if layer in self.sw_layers else 0

    def skip_mask(self) -> np.ndarray:
        m = np.zeros(self.num_layers, dtype=np.uint8)
        if self.skip_sw:
            for l in self.sw_layers:
                m[l] = 1
        return m


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    batch: int
    seq_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seed: int
    scale_mode: str = "amax"
    causal: bool = True

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


# The five workloads, numbered as listed; workload i uses seed i-1.
WORKLOADS = {
    1: DecodeWorkload("decode-1L-b1-h32x8-d128-t4096", 1, 1, 32, 8, 128, 4096, 4096, seed=0,
                      scale_mode="unit", k_outliers=4),
    2: DecodeWorkload("llama8b-decode-32L-b8-h32x8-d128-t16k-24k", 32, 8, 32, 8, 128, 16384, 24576,
                      seed=1, scale_mode="amax", k_outliers=4),
    3: DecodeWorkload("gptoss20b-hybrid-24L-b8-h64x8-d64-t8k-32k-sw128", 24, 8, 64, 8, 64, 8192, 32768,
                      seed=2, scale_mode="amax", window=128, sw_layers=tuple(range(1, 24, 2)),
                      skip_sw=True),
    4: DecodeWorkload("needle-1L-b1-h64x8-d128-t131072", 1, 1, 64, 8, 128, 131072, 131072, seed=3,
                      scale_mode="unit", needle=True, prefill_chunk=4096),
    5: PrefillWorkload("prefill-b4-t32768-h8x1-d256-causal", 4, 32768, 8, 1, 256, seed=4),
}


# ----------------------------------------------------------------------------- basic draws

def randn_bf16(shape, seed: int, layer: int, kind: str, device="cpu") -> torch.Tensor:
    g = _gen(seed, layer, kind, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def context_lengths(batch: int, lo: int, hi: int, seed: int) -> np.ndarray:
    g = _gen(seed, 0, "ctx", "cpu")
    if lo == hi:
        return np.full(batch, lo, dtype=np.int32)
    return torch.randint(lo, hi + 1, (batch,), generator=g).numpy().astype(np.int32)


def block_table(ctx: Sequence[int], seed: int, block_size: int = BLOCK_SIZE, extra_blocks: int = 0):
    """Return (table int32 [B][max_blocks], num_blocks).

    Physical blocks are a seeded permutation of range(num_blocks); unused
    entries are -1 so that a stray read is caught by the kernels' bounds check.
    """
    nb_seq = [(int(t) + block_size - 1) // block_size for t in ctx]
    total = sum(nb_seq)
    num_blocks = total + extra_blocks
    max_blocks = max(max(nb_seq), 1)
    g = _gen(seed, 0, "table", "cpu")
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    table = np.full((len(ctx), max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nb_seq):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, num_blocks


def slot_mapping(table: np.ndarray, ctx: Sequence[int], block_size: int = BLOCK_SIZE,
                 positions: Optional[Sequence[Sequence[int]]] = None) -> np.ndarray:
    """Physical slots (int64) of the given positions (default: every position of every
    sequence, sequence-major), slot = table[b][pos // bs] * bs + pos % bs."""
    out = []
    for b, t in enumerate(ctx):
        pos = np.arange(int(t)) if positions is None else np.asarray(positions[b], dtype=np.int64)
        out.append(table[b, pos // block_size].astype(np.int64) * block_size + pos % block_size)
    return np.concatenate(out) if out else np.zeros(0, dtype=np.int64)


def outlier_channels(seed: int, layer: int, num_kv_heads: int, head_dim: int, n: int) -> np.ndarray:
    """[Hkv][n] channel indices of the x8 K outliers for one layer."""
    g = _gen(seed, layer, "outlier", "cpu")
    return np.stack([torch.randperm(head_dim, generator=g)[:n].numpy() for _ in range(num_kv_heads)])


def amax_scales(x: torch.Tensor, head_axis: int) -> torch.Tensor:
    """amax/448 per head (float64 amax, one rounding to float32).  The result is an
    input to both the kernels and the oracle."""
    xf = x.abs().to(torch.float64)
    dims = [d for d in range(x.dim()) if d != head_axis]
    amax = xf.amax(dim=dims) if dims else xf
    s = (amax / E4M3_MAX).to(torch.float32)
    return torch.where(s > 0, s, torch.ones_like(s))


# ----------------------------------------------------------------------------- decode layers

@dataclasses.dataclass
class DecodeLayerData:
    """bf16 inputs of one decode layer.

    k, v: [sum_b T_b][Hkv][D] in sequence-major token order (token t of sequence b at
    row ``cu[b] + t``); q: [B][Hq][D], the query of the current (last) position.
    Scales are float32 ([1] or per head).
    """

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    q_scale: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor
    needle_pos: Optional[int] = None


def decode_layer(w: DecodeWorkload, layer: int, ctx: np.ndarray, device="cpu") -> DecodeLayerData:
    n_tok = int(np.sum(ctx))
    Hkv, Hq, D = w.num_kv_heads, w.num_q_heads, w.head_dim
    q = randn_bf16((w.batch, Hq, D), w.seed, layer, "q", device)
    kf = torch.randn((n_tok, Hkv, D), generator=_gen(w.seed, layer, "k", device), device=device,
                     dtype=torch.float32)
    if w.k_outliers:
        ch = outlier_channels(w.seed, layer, Hkv, D, w.k_outliers)
        for h in range(Hkv):
            idx = torch.as_tensor(ch[h], device=device, dtype=torch.long)
            kf[:, h, idx] *= 8.0
    needle_pos = None
    if w.needle:
        g = _gen(w.seed, layer, "needle", "cpu")
        hi = max(int(ctx[0]) - max(w.prefill_chunk, 1), 1)
        needle_pos = int(torch.randint(0, hi, (1,), generator=g).item())
        for h in range(Hkv):
            qv = q[0, h * w.group].to(torch.float32)
            kf[needle_pos, h] = 4.0 * math.sqrt(D) * qv / qv.norm()
    k = kf.to(torch.bfloat16)
    del kf
    v = randn_bf16((n_tok, Hkv, D), w.seed, layer, "v", device)
    if w.scale_mode == "unit":
        one = torch.ones(1, dtype=torch.float32, device=device)
        qs, ks, vs = one, one.clone(), one.clone()
    else:
        qs = amax_scales(q, 1)
        ks = amax_scales(k, 1)
        vs = amax_scales(v, 1)
    return DecodeLayerData(q, k, v, qs, ks, vs, needle_pos)


def prefill_query(w: DecodeWorkload, layer: int, device="cpu") -> torch.Tensor:
    """[chunk][Hq][D] bf16 queries of the prefill chunk over a decode workload's cache."""
    return randn_bf16((w.prefill_chunk, w.num_q_heads, w.head_dim), w.seed, layer, "qp", device)


@dataclasses.dataclass
class PrefillData:
    q: torch.Tensor   # [B*L][Hq][D]
    k: torch.Tensor   # [B*L][Hkv][D]
    v: torch.Tensor
    q_scale: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor


def prefill_data(w: PrefillWorkload, device="cpu", seq_len: Optional[int] = None,
                 batch: Optional[int] = None) -> PrefillData:
    L = w.seq_len if seq_len is None else seq_len
    B = w.batch if batch is None else batch
    q = randn_bf16((B * L, w.num_q_heads, w.head_dim), w.seed, 0, "q", device)
    k = randn_bf16((B * L, w.num_kv_heads, w.head_dim), w.seed, 0, "k", device)
    v = randn_bf16((B * L, w.num_kv_heads, w.head_dim), w.seed, 0, "v", device)
    if w.scale_mode == "unit":
        one = torch.ones(1, dtype=torch.float32, device=device)
        return PrefillData(q, k, v, one, one.clone(), one.clone())
    return PrefillData(q, k, v, amax_scales(q, 1), amax_scales(k, 1), amax_scales(v, 1))


# ----------------------------------------------------------------------------- conversions

def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor (host copy)."""
    return t.detach().cpu().to(torch.float32).numpy().astype(np.float64)
