"""Python binding of libfp8kv.so (FP8 KV-cache quantisation and FP8 attention, sm_103a).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (used for device memory and streams); the
C entry points receive their raw pointers.  The binding has the C ABI's names:
``kv_quant_cache``, ``fp8_decode_attn``, ``fp8_prefill_attn`` and the size queries.

The library must have been built (``python -m fp8_kv_cache_quant_gb300.build`` or
``__graft_entry__.build()``); importing the binding does not load it, calling an
entry point without it raises ``RuntimeError``.  There is no fallback path.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8kv.so")

OK, INVALID_ARG, UNSUPPORTED, CUDA_ERROR = 0, 1, 2, 3
SCALE_PER_TENSOR, SCALE_PER_HEAD = 0, 1
KV_E4M3, KV_E5M2 = 0, 1
FAULT_BLOCK_ID, FAULT_SLOT, FAULT_CONTEXT, FAULT_TIMEOUT, FAULT_QLEN, FAULT_WORKSPACE = 1, 2, 4, 8, 16, 32

# Entry points declared by include/fp8kv.h (checked by the tests).
EXPORTS = (
    "fkv_status_string", "fkv_version", "kv_quant_cache", "fp8_decode_attn_workspace_size",
    "fp8_decode_attn_num_splits", "fp8_decode_attn", "fkv_prefill_block_n", "fp8_prefill_attn",
    "fp8_decode_attn_noalloc", "fp8_decode_attn_split_blocks", "fkv_decode_block_n", "kv_quant_cache_clips",
    "fp8_decode_step", "fkv_set_decode_wait_limit_ns",
)
NOALLOC_WORKSPACE_BYTES = 16 << 20


class FkvError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


class _LayerCache(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_format", ctypes.c_int32)]


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libfp8kv.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libfp8kv.so not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    c_i32, c_vp, c_f, c_sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
    lib.fkv_status_string.restype = ctypes.c_char_p
    lib.fkv_status_string.argtypes = [ctypes.c_int]
    lib.fkv_version.restype = c_i32
    lib.fkv_set_decode_wait_limit_ns.restype = None
    lib.fkv_set_decode_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.kv_quant_cache.restype = ctypes.c_int
    lib.kv_quant_cache.argtypes = [c_vp, c_vp, c_vp, c_i32, _LayerCache, c_vp, c_vp, ctypes.c_int, c_i32, c_vp,
                                   c_i32, c_vp, c_vp]
    lib.kv_quant_cache_clips.restype = ctypes.c_int
    lib.kv_quant_cache_clips.argtypes = [c_vp, c_vp, c_vp, c_i32, _LayerCache, c_vp, c_vp, ctypes.c_int, c_i32, c_vp,
                                         c_i32, c_vp, c_vp, c_vp]
    lib.fp8_decode_attn_workspace_size.restype = c_sz
    lib.fp8_decode_attn_workspace_size.argtypes = [c_i32] * 7
    lib.fp8_decode_attn_num_splits.restype = c_i32
    lib.fp8_decode_attn_num_splits.argtypes = [c_i32] * 7
    lib.fp8_decode_attn_split_blocks.restype = c_i32
    lib.fp8_decode_attn_split_blocks.argtypes = [c_i32] * 7
    lib.fkv_decode_block_n.restype = c_i32
    lib.fkv_decode_block_n.argtypes = [c_i32, c_i32]
    lib.fp8_decode_attn.restype = ctypes.c_int
    lib.fp8_decode_attn.argtypes = [c_vp, c_i32, c_i32, _LayerCache, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp,
                                    ctypes.c_int, c_f, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, c_sz, c_i32, c_vp,
                                    c_vp]
    lib.fp8_decode_step.restype = ctypes.c_int
    lib.fp8_decode_step.argtypes = [c_vp, c_vp] + lib.fp8_decode_attn.argtypes
    lib.fp8_decode_attn_noalloc.restype = ctypes.c_int
    lib.fp8_decode_attn_noalloc.argtypes = [c_vp, c_i32, c_i32, _LayerCache, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp,
                                            ctypes.c_int, c_f, c_i32, c_i32, c_vp, c_i32, c_vp, c_i32, c_vp, c_vp]
    lib.fkv_prefill_block_n.restype = c_i32
    lib.fkv_prefill_block_n.argtypes = [c_i32]
    lib.fp8_prefill_attn.restype = ctypes.c_int
    lib.fp8_prefill_attn.argtypes = [c_vp, c_vp, c_i32, c_i32, c_i32, _LayerCache, c_vp, c_i32, c_vp, c_vp, c_vp,
                                     c_vp, ctypes.c_int, c_f, c_i32, c_i32, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp,
                                     c_vp]
    if path is None:
        _lib = lib
    return lib


def _check(fn: str, st: int):
    if st != OK:
        raise FkvError(fn, st, load_library().fkv_status_string(st).decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclasses.dataclass
class LayerCache:
    """One layer's K/V pools: uint8 (FP8 codes of ``kv_format``: KV_E4M3 or KV_E5M2) or
    bfloat16 tensors [num_blocks][Hkv][16][D]."""

    k_cache: torch.Tensor
    v_cache: torch.Tensor
    kv_format: int = 0

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def num_kv_heads(self):
        return self.k_cache.shape[1]

    @property
    def block_size(self):
        return self.k_cache.shape[2]

    @property
    def head_dim(self):
        return self.k_cache.shape[3]

    def c(self) -> _LayerCache:
        return _LayerCache(self.k_cache.data_ptr(), self.v_cache.data_ptr(), self.num_blocks, self.block_size,
                           self.num_kv_heads, self.head_dim, self.kv_format)

    @staticmethod
    def empty(num_blocks, num_kv_heads, head_dim, bf16=False, device="cuda", block_size=16, kv_format=0):
        dt = torch.bfloat16 if bf16 else torch.uint8
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        return LayerCache(torch.empty(shape, dtype=dt, device=device), torch.empty(shape, dtype=dt, device=device),
                          kv_format)


def _mask_arg(skip_layer_mask):
    if skip_layer_mask is None:
        return None, 0, None
    arr = np.ascontiguousarray(np.asarray(skip_layer_mask, dtype=np.uint8))
    return arr.ctypes.data, int(arr.size), arr   # keep arr alive in the caller


def kv_quant_cache(k, v, slot_mapping, cache: LayerCache, k_scale=None, v_scale=None, gran=SCALE_PER_TENSOR,
                   layer=0, skip_layer_mask=None, fault=None, stream=None):
    lib = load_library()
    mp, nl, keep = _mask_arg(skip_layer_mask)
    st = lib.kv_quant_cache(_ptr(k), _ptr(v), _ptr(slot_mapping), int(k.shape[0]), cache.c(), _ptr(k_scale),
                            _ptr(v_scale), int(gran), int(layer), mp, nl, _ptr(fault), _stream(stream))
    del keep
    _check("kv_quant_cache", st)


def kv_quant_cache_clips(k, v, slot_mapping, cache: LayerCache, k_scale, v_scale, gran=SCALE_PER_TENSOR,
                         clip_counts=None, layer=0, skip_layer_mask=None, fault=None, stream=None):
    """kv_quant_cache that also adds the numbers of clipped K and V elements to
    ``clip_counts`` (device int64 [2], created zeroed when None); returns it."""
    lib = load_library()
    if clip_counts is None:
        clip_counts = torch.zeros(2, dtype=torch.int64, device=k.device)
    mp, nl, keep = _mask_arg(skip_layer_mask)
    st = lib.kv_quant_cache_clips(_ptr(k), _ptr(v), _ptr(slot_mapping), int(k.shape[0]), cache.c(), _ptr(k_scale),
                                  _ptr(v_scale), int(gran), int(layer), mp, nl, _ptr(clip_counts), _ptr(fault),
                                  _stream(stream))
    del keep
    _check("kv_quant_cache_clips", st)
    return clip_counts


def fp8_decode_attn_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, window=0,
                                   num_splits=0) -> int:
    return int(load_library().fp8_decode_attn_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                              max_blocks, window, num_splits))


def fp8_decode_attn_num_splits(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, window=0,
                               num_splits=0) -> int:
    return int(load_library().fp8_decode_attn_num_splits(batch, num_q_heads, num_kv_heads, head_dim, max_blocks,
                                                          window, num_splits))


def fp8_decode_attn_split_blocks(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, window=0,
                                 num_splits=0) -> int:
    return int(load_library().fp8_decode_attn_split_blocks(batch, num_q_heads, num_kv_heads, head_dim, max_blocks,
                                                            window, num_splits))


def fkv_decode_block_n(head_dim: int, bf16_layer: bool = False, kv_format: int = 0) -> int:
    kind = 1 if bf16_layer else (2 if kv_format == KV_E5M2 else 0)
    return int(load_library().fkv_decode_block_n(head_dim, kind))


def decode_workspace(batch, num_q_heads, cache: LayerCache, max_blocks, window=0, num_splits=0, device="cuda"):
    """A zero-filled decode workspace (the split counters at its start must be zero when a
    call begins; every call leaves them zero)."""
    n = fp8_decode_attn_workspace_size(batch, num_q_heads, cache.num_kv_heads, cache.head_dim, max_blocks,
                                       window, num_splits)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def fp8_decode_attn(q, cache: LayerCache, block_table, context_lens, q_scale=None, k_scale=None, v_scale=None,
                    gran=SCALE_PER_TENSOR, softmax_scale=0.0, window=0, layer=0, skip_layer_mask=None, out=None,
                    workspace=None, num_splits=0, fault=None, stream=None):
    lib = load_library()
    B, Hq, D = q.shape
    max_blocks = int(block_table.shape[1])
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, cache, max_blocks, window, num_splits, q.device)
    mp, nl, keep = _mask_arg(skip_layer_mask)
    st = lib.fp8_decode_attn(_ptr(q), B, Hq, cache.c(), _ptr(block_table), max_blocks, _ptr(context_lens),
                             _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), int(gran), float(softmax_scale),
                             int(window), int(layer), mp, nl, _ptr(out), _ptr(workspace),
                             int(workspace.numel() * workspace.element_size()), int(num_splits), _ptr(fault),
                             _stream(stream))
    del keep
    _check("fp8_decode_attn", st)
    return out


def fp8_decode_step(k_new, v_new, q, cache: LayerCache, block_table, context_lens, q_scale=None, k_scale=None,
                    v_scale=None, gran=SCALE_PER_TENSOR, softmax_scale=0.0, window=0, layer=0, skip_layer_mask=None,
                    out=None, workspace=None, num_splits=0, fault=None, stream=None):
    """kv_quant_cache of the current token (k_new, v_new: bf16 [batch][num_kv_heads][head_dim], written at
    position context_lens[b] - 1) and fp8_decode_attn in one launch (e4m3 layers)."""
    lib = load_library()
    B, Hq, D = q.shape
    max_blocks = int(block_table.shape[1])
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, cache, max_blocks, window, num_splits, q.device)
    mp, nl, keep = _mask_arg(skip_layer_mask)
    st = lib.fp8_decode_step(_ptr(k_new), _ptr(v_new), _ptr(q), B, Hq, cache.c(), _ptr(block_table), max_blocks,
                             _ptr(context_lens), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), int(gran),
                             float(softmax_scale), int(window), int(layer), mp, nl, _ptr(out), _ptr(workspace),
                             int(workspace.numel() * workspace.element_size()), int(num_splits), _ptr(fault),
                             _stream(stream))
    del keep
    _check("fp8_decode_step", st)
    return out


def fp8_decode_attn_noalloc(q, cache: LayerCache, block_table, context_lens, q_scale=None, k_scale=None,
                            v_scale=None, gran=SCALE_PER_TENSOR, softmax_scale=0.0, window=0, layer=0,
                            skip_layer_mask=None, out=None, num_splits=0, fault=None, stream=None):
    """fp8_decode_attn without a workspace: the library's fixed device scratch is used
    (see include/fp8kv.h for its size limit and the sharing rule)."""
    lib = load_library()
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    mp, nl, keep = _mask_arg(skip_layer_mask)
    st = lib.fp8_decode_attn_noalloc(_ptr(q), B, Hq, cache.c(), _ptr(block_table), int(block_table.shape[1]),
                                     _ptr(context_lens), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), int(gran),
                                     float(softmax_scale), int(window), int(layer), mp, nl, _ptr(out),
                                     int(num_splits), _ptr(fault), _stream(stream))
    del keep
    _check("fp8_decode_attn_noalloc", st)
    return out


def fkv_prefill_block_n(head_dim: int) -> int:
    return int(load_library().fkv_prefill_block_n(head_dim))


def fp8_prefill_attn(q, cu_seqlens_q, max_q_len, cache: LayerCache, block_table, context_lens, q_scale=None,
                     k_scale=None, v_scale=None, gran=SCALE_PER_TENSOR, softmax_scale=0.0, causal=True, window=0,
                     promote_every=1, layer=0, skip_layer_mask=None, out=None, fault=None, stream=None):
    lib = load_library()
    N, Hq, D = q.shape
    B = int(cu_seqlens_q.shape[0]) - 1
    if out is None:
        out = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=q.device)
    mp, nl, keep = _mask_arg(skip_layer_mask)
    st = lib.fp8_prefill_attn(_ptr(q), _ptr(cu_seqlens_q), B, Hq, int(max_q_len), cache.c(), _ptr(block_table),
                              int(block_table.shape[1]), _ptr(context_lens), _ptr(q_scale), _ptr(k_scale),
                              _ptr(v_scale), int(gran), float(softmax_scale), int(bool(causal)), int(window),
                              int(promote_every), int(layer), mp, nl, _ptr(out), _ptr(fault), _stream(stream))
    del keep
    _check("fp8_prefill_attn", st)
    return out
