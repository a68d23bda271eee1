"""Decode and prefill attention over an FP8 (or bf16) paged KV cache, in float64.

What is computed (vLLM blog "FP8 KV-Cache and Attention quantization in vLLM"):
  * 引言: with ``--kv-cache-dtype fp8`` the KV cache is stored in e4m3 and the whole
    attention runs in FP8, the QK and Score*V products included;
  * "Kernel 与 vLLM 改进", "Per-Head Scales": one scale per KV head;
    "Query Quantization Fusion": the query is quantised to FP8 as well;
  * "单请求 Benchmark": FlashAttention-style attention with online softmax
    rescaling; "Kernel 与 vLLM 改进", "Two-level accumulation": the partial Score*V
    accumulation of each tile is added into a true FP32 accumulator.

Readings where the pages are silent (each is exercised by the tests):
  R5  query head h uses KV head h // G (contiguous GQA grouping);
  R6  a window W keeps exactly the last W keys, the current one included;
  R7  decode quantises Q with its scale (1.0 when uncalibrated);
  R8  softmax scale 1/sqrt(D);
  R9  decode keeps P exact (``p_quant=False``), or, for a decode whose Score*V product
      runs on FP8 tensor cores (``p_quant=True``), rounds P per key tile as prefill does
      (R11) with the tiles of the kernel's splits (R23);
  R10 the prefill softmax denominator sums the unrounded p;
  R11 prefill rounds P to e4m3 as e4m3(p * 448) and divides by 448 again;
  R13 prefill query i of a sequence with context T and Lq queries sits at absolute
      position T - Lq + i (the chunk is the tail of the context);
  R25 an e5m2 layer stores K and V as e5m2 codes (scales as for e4m3) and attends with
      the bf16 query and exact P: the codes are dequantised, nothing else is rounded;
  R23 a split-K decode with FP8 P splits the key range [lo, T) into runs of
      ``split_blocks`` pool blocks starting at block lo // block_size; each split walks
      its keys in tiles of ``block_n`` starting at its first block, with its own running
      maximum, and the splits' (acc, m, l) are merged exactly.

With exact P the decode oracle computes the unsplit softmax (split-K is exactly the same
sum).
The prefill oracle walks the keys in the kernel's tiles because the e4m3 rounding of
p depends on the running maximum at each tile; with ``p_quant=False`` it is the plain
softmax definition.
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3, e5m2
from .kvcache import head_scale


def _gather(pool, table_row, positions, g, block_size):
    blk = table_row[positions // block_size]
    off = positions % block_size
    return pool[blk, g, off, :]


def _dequant_rows(rows, scale, fp8: bool, fmt: str = "e4m3"):
    if fp8:
        return (e5m2 if fmt == "e5m2" else e4m3).decode(rows) * scale
    return np.asarray(rows, dtype=np.float64)


def softmax_attend(qv, K, V, tau):
    """o = softmax(tau * K q) V for one query vector, max-subtracted, float64."""
    s = (K @ qv) * tau
    m = np.max(s)
    w = np.exp(s - m)
    w /= np.sum(w)
    return w @ V, w


def p_rounding_bound(qv, K, V, tau):
    """Element-wise bound on how far an attention that rounds P to e4m3 can sit from the
    exact softmax result, for one query vector over dequantised K, V [T][D].

    The FP8 Score*V product (vLLM blog, 引言; "Kernel 与 vLLM 改进", Two-level
    accumulation) multiplies V by P8 = e4m3(p * 448) with p = e^(s - m') taken against a
    running maximum m' <= M = max_j s_j, and divides by 448 again; the denominator sums
    the unrounded p (R10, R11).  e4m3 has 3 mantissa bits, so a code >= 2^-6 (normal)
    is within 2^-4 relatively of p * 448, a subnormal code (spacing 2^-9) within 2^-10
    absolutely, and p * 448 <= 448 never saturates.  Rescaled to the global maximum
    (factor e^(m' - M) <= 1), every rounded weight satisfies
        |p^_j - p_j| <= max(2^-4 p_j, 2^-10 / 448),   p_j = e^(s_j - M),
    hence, with l = sum_j p_j and o the exact output,
        |o^_d - o_d| <= B_d = sum_j max(2^-4 p_j, 2^-10 / 448) |v_jd| / l.
    Returns (o, B), both float64 [D]; the bound holds for every split and tile plan."""
    s = (np.asarray(K, np.float64) @ np.asarray(qv, np.float64)) * tau
    p = np.exp(s - np.max(s))
    l = np.sum(p)
    Va = np.abs(np.asarray(V, np.float64))
    eps = np.maximum(2.0 ** -4 * p, 2.0 ** -10 / 448.0)
    return (p @ V) / l, (eps @ Va) / l


def split_decode(qv, K, V, T, lo, tau, *, split_blocks, block_n, p_quant, block_size=16):
    """One query over keys lo .. T-1 (dequantised K, V [T - lo][D]) as a split-K decode
    (R23): splits of ``split_blocks`` blocks from block lo // block_size, each walked in
    tiles of ``block_n`` from its first block with its own running maximum (P rounded
    as e4m3(p * 448) / 448 when ``p_quant``), then merged:
    o = sum_s e^(m_s - M) acc_s / sum_s e^(m_s - M) l_s,  M = max_s m_s."""
    blk0, blk1 = lo // block_size, (T + block_size - 1) // block_size
    qpos = np.array([T - 1])
    accs, ms, ls = [], [], []
    for b0 in range(blk0, blk1, split_blocks):
        b1 = min(b0 + split_blocks, blk1)
        a, z = max(lo, b0 * block_size), min(T, b1 * block_size)
        if z <= a:
            continue
        acc, m, l = _tile_walk(np.asarray(qv)[None, :], K[a - lo:z - lo], V[a - lo:z - lo], qpos, a, block_n, tau,
                               p_quant, tile0=b0 * block_size, state=True)
        accs.append(acc[0]); ms.append(m[0]); ls.append(l[0])
    if not ms:
        return np.zeros(V.shape[1])
    M = max(ms)
    w = [math.exp(mi - M) for mi in ms]
    num = sum(wi * ai for wi, ai in zip(w, accs))
    den = sum(wi * li for wi, li in zip(w, ls))
    return num / den


def decode_attention(q, k_pool, v_pool, block_table, context_lens, q_scale, k_scale, v_scale, *,
                     fp8: bool = True, softmax_scale: float = 0.0, window: int = 0, block_size: int = 16,
                     p_quant: bool = False, split_blocks: int = 0, block_n: int = 128, fmt: str = "e4m3",
                     p_bound: bool = False):
    """Paged decode attention, one query per sequence.

    q: float64 [B][Hq][D] (bf16 values).  k_pool / v_pool: uint8 e4m3 codes
    ``[nb][Hkv][bs][D]`` when ``fp8``, else float64 values of the bf16 pool.
    context_lens[b] counts every key of sequence b, the current token included.
    Returns float64 [B][Hq][D]; a sequence with no key gives a zero row.
    ``split_blocks`` > 0 computes it as the split-K decode of R23 (``p_quant`` rounds P,
    on e4m3 layers only); 0 is the plain softmax.  ``fmt`` "e5m2" reads e5m2 pools with
    the bf16 query and exact P (R25).  ``p_bound`` returns (plain softmax result, the
    element-wise bound of ``p_rounding_bound``), both [B][Hq][D].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    tau = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(D)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    bound = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        T = int(context_lens[b])
        lo = max(0, T - window) if window > 0 else 0
        if T - lo <= 0:
            continue
        pos = np.arange(lo, T, dtype=np.int64)
        for g in range(Hkv):
            K = _dequant_rows(_gather(k_pool, block_table[b], pos, g, block_size), head_scale(k_scale, g), fp8, fmt)
            V = _dequant_rows(_gather(v_pool, block_table[b], pos, g, block_size), head_scale(v_scale, g), fp8, fmt)
            for h in range(g * G, (g + 1) * G):
                if fp8 and fmt == "e4m3":
                    qs = head_scale(q_scale, h)
                    qv = e4m3.decode(e4m3.quantize(q[b, h], qs)) * qs
                else:
                    qv = q[b, h]
                if p_bound:
                    out[b, h], bound[b, h] = p_rounding_bound(qv, K, V, tau)
                elif split_blocks > 0:
                    out[b, h] = split_decode(qv, K, V, T, lo, tau, split_blocks=split_blocks, block_n=block_n,
                                             p_quant=p_quant and fp8 and fmt == "e4m3", block_size=block_size)
                else:
                    out[b, h], _ = softmax_attend(qv, K, V, tau)
    return (out, bound) if p_bound else out


def decode_attention_contiguous(q_b, k_seq, v_seq, q_scale, k_scale, v_scale, *, fp8=True,
                                softmax_scale=0.0, window=0, heads=None, p_quant=False, split_blocks=0,
                                block_n=128, p_bound=False):
    """Decode attention of ONE sequence from its contiguous bf16 K/V ([T][Hkv][D],
    float64 values): the oracle quantises K/V itself with the same rule as the cache
    write, then attends (as the split-K decode of R23 when ``split_blocks`` > 0).  Used
    at full workload sizes on sampled sequences/heads.
    Returns {h: float64[D]} for the requested query heads (default: all); with
    ``p_bound`` {h: (o, B)}: the exact softmax result and the bound of
    ``p_rounding_bound`` on an attention that rounds P to e4m3."""
    Hq, D = q_b.shape
    T, Hkv, _ = k_seq.shape
    G = Hq // Hkv
    tau = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(D)
    lo = max(0, T - window) if window > 0 else 0
    heads = range(Hq) if heads is None else heads
    res = {}
    cache = {}
    for h in heads:
        g = h // G
        if g not in cache:
            ks, vs = head_scale(k_scale, g), head_scale(v_scale, g)
            Kb, Vb = k_seq[lo:T, g], v_seq[lo:T, g]
            if fp8:
                K = e4m3.decode(e4m3.quantize(Kb, ks)) * ks
                V = e4m3.decode(e4m3.quantize(Vb, vs)) * vs
            else:
                K, V = np.asarray(Kb, np.float64), np.asarray(Vb, np.float64)
            cache = {g: (K, V)}
        K, V = cache[g]
        if T - lo <= 0:
            res[h] = (np.zeros(D), np.zeros(D)) if p_bound else np.zeros(D)
            continue
        if fp8:
            qs = head_scale(q_scale, h)
            qv = e4m3.decode(e4m3.quantize(q_b[h], qs)) * qs
        else:
            qv = q_b[h]
        if p_bound:
            res[h] = p_rounding_bound(qv, K, V, tau)
        elif split_blocks > 0:
            res[h] = split_decode(qv, K, V, T, lo, tau, split_blocks=split_blocks, block_n=block_n,
                                  p_quant=p_quant and fp8)
        else:
            res[h], _ = softmax_attend(qv, K, V, tau)
    return res


def _tile_walk(Qt, K, V, qpos, kpos0, block_n, tau, p_quant, window=0, tile0=0, state=False):
    """Online softmax over key tiles for a set of query rows of one head.

    Qt: [R][D] dequantised queries at absolute positions qpos [R]; K, V: [T][D]
    dequantised keys/values at absolute positions kpos0 .. kpos0+T-1 (kpos0 >= tile0).
    Tiles are the key ranges [tile0 + t*block_n, tile0 + (t+1)*block_n).  Row r sees
    keys <= qpos[r].
    For each tile: m_t = max(m_{t-1}, tile max); p = exp(s - m_t);
    l = l e^{m_{t-1}-m_t} + sum p (unrounded p, R10);
    acc = acc e^{m_{t-1}-m_t} + sum e4m3(p*448)/448 * v (R11, two-level: the tile's
    partial is added into the running float accumulator).
    Returns acc / l, or with ``state`` the unnormalised (acc, m, l) (natural-log max).
    """
    R, D = Qt.shape
    T = K.shape[0]
    S = (Qt @ K.T) * tau                      # [R][T]
    kabs = kpos0 + np.arange(T)
    valid = kabs[None, :] <= qpos[:, None]
    if window > 0:
        valid &= kabs[None, :] >= (qpos[:, None] - window + 1)
    S = np.where(valid, S, -np.inf)
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    acc = np.zeros((R, V.shape[1]))
    t_first = (kpos0 - tile0) // block_n
    t_last = (kpos0 + T - 1 - tile0) // block_n
    for t in range(t_first, t_last + 1):
        a = max(tile0 + t * block_n, kpos0) - kpos0
        b = min(tile0 + (t + 1) * block_n, kpos0 + T) - kpos0
        st = S[:, a:b]
        tmax = np.max(st, axis=1)
        m_new = np.maximum(m, tmax)
        live = np.isfinite(m_new)
        m_safe = np.where(live, m_new, 0.0)
        alpha = np.where(np.isfinite(m), np.exp(np.where(live, m - m_safe, 0.0)), 0.0)
        p = np.exp(st - m_safe[:, None])
        p = np.where(np.isfinite(st), p, 0.0)
        l = l * alpha + p.sum(axis=1)
        if p_quant:
            pq = e4m3.decode(e4m3.encode(e4m3.fl32(e4m3.fl32(p) * 448.0))) / 448.0
        else:
            pq = p
        acc = acc * alpha[:, None] + pq @ V[a:b]
        m = np.where(live, m_new, m)
    if state:
        return acc, m, l
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return out


def prefill_attention(q, cu_seqlens, k_seq_list, v_seq_list, q_scale, k_scale, v_scale, *, block_n: int,
                      fp8: bool = True, p_quant: bool = True, softmax_scale: float = 0.0,
                      causal: bool = True, rows=None, window: int = 0):
    """Prefill (chunked) attention with the kernel's tile walk.

    q: float64 [sum Lq][Hq][D]; cu_seqlens: [B+1]; k_seq_list[b] / v_seq_list[b]:
    float64 [T_b][Hkv][D] bf16 values of the whole context of sequence b (the oracle
    quantises them with the cache-write rule).  ``rows`` optionally restricts the
    computed query rows to a list of global row indices (others are NaN).
    Non-causal means every row sees the whole context.  A window W > 0 keeps, for the row
    at position p, only keys [p - W + 1, p] (R6: the last W keys, its own included).
    Returns float64 [sum Lq][Hq][D].
    """
    q = np.asarray(q, dtype=np.float64)
    N, Hq, D = q.shape
    tau = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(D)
    out = np.full((N, Hq, D), np.nan)
    want = None if rows is None else set(int(r) for r in rows)
    for b in range(len(cu_seqlens) - 1):
        r0, r1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        Lq = r1 - r0
        if Lq == 0:
            continue
        kb, vb = k_seq_list[b], v_seq_list[b]
        T, Hkv, _ = kb.shape
        G = Hq // Hkv
        sel = np.arange(r0, r1) if want is None else np.array(sorted(r for r in want if r0 <= r < r1), dtype=np.int64)
        if sel.size == 0:
            continue
        qpos = (T - Lq) + (sel - r0) if causal else np.full(sel.size, T - 1)
        for g in range(Hkv):
            ks, vs = head_scale(k_scale, g), head_scale(v_scale, g)
            if fp8:
                K = e4m3.decode(e4m3.quantize(kb[:, g], ks)) * ks
                V = e4m3.decode(e4m3.quantize(vb[:, g], vs)) * vs
            else:
                K, V = kb[:, g], vb[:, g]
            kmax = int(qpos.max()) + 1
            for h in range(g * G, (g + 1) * G):
                if fp8:
                    qs = head_scale(q_scale, h)
                    Qt = e4m3.decode(e4m3.quantize(q[sel, h], qs)) * qs
                else:
                    Qt = q[sel, h]
                out[sel, h] = _tile_walk(Qt, K[:kmax], V[:kmax], qpos, 0, block_n, tau, p_quant and fp8, window)
    return out
