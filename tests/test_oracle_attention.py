"""Pins of the oracle's decode and prefill attention (CPU only).

Each check comes from outside the oracle's own formulas: a pure-Python loop
implementation on tiny inputs, closed forms (identical keys, one dominant key, a
single key, empty context), invariants (weights sum to one, block-table
permutation), torch's float64 scaled_dot_product_attention for the unquantised
special case, and a hand-worked two-tile example of the P rounding with running-max
rescaling.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, e4m3, kvcache

BS = 16


def _paged(K, V, T_list, rng, fp8, ks, vs, bs=BS):
    """Build pools and a shuffled block table with the oracle's own cache write."""
    B = len(T_list)
    Hkv, D = K[0].shape[1], K[0].shape[2]
    nblk = [(t + bs - 1) // bs for t in T_list]
    nb = sum(nblk) + 3
    perm = rng.permutation(nb)
    table = np.full((B, max(max(nblk), 1)), -1, dtype=np.int64)
    off = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += nblk[b]
    if fp8:
        kp = np.full((nb, Hkv, bs, D), 0x5A, np.uint8)
        vp = np.full((nb, Hkv, bs, D), 0x5A, np.uint8)
    else:
        kp = np.zeros((nb, Hkv, bs, D))
        vp = np.zeros((nb, Hkv, bs, D))
    for b in range(B):
        pos = np.arange(T_list[b])
        slots = table[b, pos // bs] * bs + pos % bs
        kvcache.cache_write(K[b], V[b], slots, kp, vp, ks, vs, skip=not fp8, block_size=bs)
    return kp, vp, table


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def _loop_decode(q, K, V, qs, ks, vs, fp8, tau, window=0):
    """Pure-Python loops (no numpy reductions) for one sequence, all heads."""
    Hq, D = len(q), len(q[0])
    T, Hkv = len(K), len(K[0])
    G = Hq // Hkv
    lo = max(0, T - window) if window else 0
    out = []
    for h in range(Hq):
        g = h // G
        if fp8:
            qv = [float(e4m3.decode(e4m3.quantize(np.array([q[h][d]]), kvcache.head_scale(qs, h)))[0])
                  * kvcache.head_scale(qs, h) for d in range(D)]
        else:
            qv = [q[h][d] for d in range(D)]
        scores, vals = [], []
        for j in range(lo, T):
            if fp8:
                kj = [float(e4m3.decode(e4m3.quantize(np.array([K[j][g][d]]), kvcache.head_scale(ks, g)))[0])
                      * kvcache.head_scale(ks, g) for d in range(D)]
                vj = [float(e4m3.decode(e4m3.quantize(np.array([V[j][g][d]]), kvcache.head_scale(vs, g)))[0])
                      * kvcache.head_scale(vs, g) for d in range(D)]
            else:
                kj, vj = list(K[j][g]), list(V[j][g])
            scores.append(sum(qv[d] * kj[d] for d in range(D)) * tau)
            vals.append(vj)
        mx = max(scores)
        w = [math.exp(s - mx) for s in scores]
        z = sum(w)
        out.append([sum(w[j] * vals[j][d] for j in range(len(w))) / z for d in range(D)])
    return np.array(out)


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("window", [0, 3])
def test_decode_matches_python_loops(fp8, window):
    rng = np.random.default_rng(10)
    Hq, Hkv, D = 4, 2, 4
    T_list = [1, 5, 8, 19]
    q = _bf16(rng.standard_normal((len(T_list), Hq, D)) * 2)
    K = [_bf16(rng.standard_normal((t, Hkv, D)) * 3) for t in T_list]
    V = [_bf16(rng.standard_normal((t, Hkv, D))) for t in T_list]
    qs = np.array([0.5, 1.0, 0.25, 2.0], np.float32)
    ks = np.array([0.75, 0.125], np.float32)
    vs = np.array([1.5, 0.5], np.float32)
    kp, vp, table = _paged(K, V, T_list, rng, fp8, ks, vs, bs=4)
    got = attention.decode_attention(q, kp, vp, table, T_list, qs, ks, vs, fp8=fp8, window=window, block_size=4)
    for b, T in enumerate(T_list):
        ref = _loop_decode(q[b], K[b], V[b], qs, ks, vs, fp8, 1 / math.sqrt(D), window)
        np.testing.assert_allclose(got[b], ref, rtol=1e-12, atol=1e-12)


def test_decode_unquantised_matches_sdpa():
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D = 3, 8, 2, 32
    T_list = [37, 64, 100]
    q = _bf16(rng.standard_normal((B, Hq, D)))
    K = [_bf16(rng.standard_normal((t, Hkv, D))) for t in T_list]
    V = [_bf16(rng.standard_normal((t, Hkv, D))) for t in T_list]
    one = np.ones(1, np.float32)
    kp, vp, table = _paged(K, V, T_list, rng, False, one, one)
    got = attention.decode_attention(q, kp, vp, table, T_list, one, one, one, fp8=False)
    for b, T in enumerate(T_list):
        qt = torch.from_numpy(q[b]).unsqueeze(1)                       # [Hq][1][D]
        kt = torch.from_numpy(K[b]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        vt = torch.from_numpy(V[b]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).squeeze(1).numpy()
        np.testing.assert_allclose(got[b], ref, rtol=1e-12, atol=1e-13)


def test_decode_closed_forms():
    D, Hkv, Hq = 8, 1, 2
    rng = np.random.default_rng(12)
    one = np.ones(1, np.float32)
    # identical keys -> mean of the values
    T = 21
    k = np.tile(_bf16(rng.standard_normal(D)), (T, Hkv, 1))
    v = _bf16(rng.standard_normal((T, Hkv, D)))
    q = _bf16(rng.standard_normal((1, Hq, D)))
    kp, vp, table = _paged([k], [v], [T], rng, True, one, one)
    o = attention.decode_attention(q, kp, vp, table, [T], one, one, one)
    vt = e4m3.decode(e4m3.quantize(v[:, 0], 1.0))
    np.testing.assert_allclose(o[0, 0], vt.mean(axis=0), rtol=1e-12, atol=1e-12)
    # one dominant key (logit gap >= 40) -> its value row
    qd = np.zeros((1, Hq, D)); qd[0, :, 0] = 16.0
    kd = np.zeros((T, Hkv, D)); kd[7, 0, 0] = 32.0          # logit 16*32/sqrt(8) = 181
    kp, vp, table = _paged([kd], [v], [T], rng, True, one, one)
    o = attention.decode_attention(qd, kp, vp, table, [T], one, one, one)
    np.testing.assert_allclose(o[0, 1], vt[7], rtol=1e-12, atol=1e-12)
    # a single key -> its value; an empty context -> zeros
    kp, vp, table = _paged([k[:1]], [v[:1]], [1], rng, True, one, one)
    o = attention.decode_attention(q, kp, vp, table, [1], one, one, one)
    np.testing.assert_allclose(o[0, 0], vt[0], rtol=0, atol=0)
    o = attention.decode_attention(q, kp, vp, table, [0], one, one, one)
    assert np.all(o == 0)
    # a window of one key keeps only the current token
    kp, vp, table = _paged([k], [v], [T], rng, True, one, one)
    o = attention.decode_attention(q, kp, vp, table, [T], one, one, one, window=1)
    np.testing.assert_allclose(o[0, 0], vt[T - 1], rtol=0, atol=0)


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(13)
    for T in (1, 7, 500):
        K = rng.standard_normal((T, 16)) * 5
        _, w = attention.softmax_attend(rng.standard_normal(16), K, rng.standard_normal((T, 16)), 0.25)
        assert abs(w.sum() - 1.0) < 1e-12


def test_gqa_grouping_is_contiguous():
    # R5: q head h reads KV head h // G.  Give every KV head a different dominant key.
    D, Hkv, G, T = 4, 4, 3, 16
    one = np.ones(1, np.float32)
    K = np.zeros((T, Hkv, D)); V = np.zeros((T, Hkv, D))
    for g in range(Hkv):
        K[g, g, 0] = 64.0
        V[g, g, :] = g + 1
    q = np.zeros((1, Hkv * G, D)); q[0, :, 0] = 8.0
    rng = np.random.default_rng(14)
    kp, vp, table = _paged([K], [V], [T], rng, True, one, one)
    o = attention.decode_attention(q, kp, vp, table, [T], one, one, one)
    for h in range(Hkv * G):
        np.testing.assert_allclose(o[0, h], np.full(D, h // G + 1), atol=1e-9)


def test_block_table_permutation_invariance():
    rng = np.random.default_rng(15)
    T_list = [50, 33]
    K = [_bf16(rng.standard_normal((t, 2, 16))) for t in T_list]
    V = [_bf16(rng.standard_normal((t, 2, 16))) for t in T_list]
    q = _bf16(rng.standard_normal((2, 4, 16)))
    one = np.ones(1, np.float32)
    outs = []
    for seed in (1, 2):
        kp, vp, table = _paged(K, V, T_list, np.random.default_rng(seed), True, one, one)
        outs.append(attention.decode_attention(q, kp, vp, table, T_list, one, one, one))
    assert np.array_equal(outs[0], outs[1])


# ----------------------------------------------------------------------------- prefill

def test_prefill_unquantised_matches_sdpa_causal_tail():
    rng = np.random.default_rng(20)
    Hq, Hkv, D = 4, 2, 16
    T_list, Lq_list = [40, 70], [40, 23]
    K = [_bf16(rng.standard_normal((t, Hkv, D))) for t in T_list]
    V = [_bf16(rng.standard_normal((t, Hkv, D))) for t in T_list]
    cu = np.concatenate([[0], np.cumsum(Lq_list)])
    q = _bf16(rng.standard_normal((cu[-1], Hq, D)))
    one = np.ones(1, np.float32)
    got = attention.prefill_attention(q, cu, K, V, one, one, one, block_n=16, fp8=False)
    for b in range(2):
        T, Lq = T_list[b], Lq_list[b]
        qt = torch.from_numpy(q[cu[b]:cu[b + 1]]).permute(1, 0, 2)
        kt = torch.from_numpy(K[b]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        vt = torch.from_numpy(V[b]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        qpos = T - Lq + np.arange(Lq)
        mask = torch.from_numpy(np.arange(T)[None, :] <= qpos[:, None])
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).permute(1, 0, 2).numpy()
        np.testing.assert_allclose(got[cu[b]:cu[b + 1]], ref, rtol=1e-11, atol=1e-12)


def test_prefill_tile_size_irrelevant_without_p_rounding():
    rng = np.random.default_rng(21)
    K = [_bf16(rng.standard_normal((300, 1, 8)))]
    V = [_bf16(rng.standard_normal((300, 1, 8)))]
    q = _bf16(rng.standard_normal((300, 2, 8)))
    one = np.ones(1, np.float32)
    a = attention.prefill_attention(q, [0, 300], K, V, one, one, one, block_n=16, p_quant=False)
    b = attention.prefill_attention(q, [0, 300], K, V, one, one, one, block_n=128, p_quant=False)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    c = attention.prefill_attention(q, [0, 300], K, V, one, one, one, block_n=128, p_quant=True)
    assert not np.allclose(a, c, rtol=1e-6, atol=0), "P rounding must change the result"


def test_prefill_two_tile_hand_example():
    # D = 1, softmax scale 1, q = 1, keys 1 then 0 (one key per tile), values 2 and 4.
    # Tile 0: m = 1, p = 1 -> e4m3(448) = 448 exactly, l = 1, acc = 2.
    # Tile 1: m stays 1, p = e^-1, p*448 = 164.8 -> nearest e4m3 is 160 (step 16 in
    # [128, 256)), l = 1 + e^-1 (unrounded p, R10), acc = 2 + (160/448)*4.
    one = np.ones(1, np.float32)
    K = [np.array([[[1.0]], [[0.0]]])]
    V = [np.array([[[2.0]], [[4.0]]])]
    q = np.array([[[1.0]], [[1.0]]])
    out = attention.prefill_attention(q, [0, 2], K, V, one, one, one, block_n=1, softmax_scale=1.0)
    expect = (2.0 + 160.0 / 448.0 * 4.0) / (1.0 + math.exp(-1.0))
    assert abs(out[1, 0, 0] - expect) < 1e-12
    assert out[0, 0, 0] == 2.0        # row 0 sees only key 0
    # reversed keys: the second tile raises the max, the first tile's partial is rescaled
    K = [np.array([[[0.0]], [[1.0]]])]
    out = attention.prefill_attention(q, [0, 2], K, V, one, one, one, block_n=1, softmax_scale=1.0)
    expect = (2.0 * math.exp(-1.0) + 4.0) / (math.exp(-1.0) + 1.0)
    assert abs(out[1, 0, 0] - expect) < 1e-12


def test_prefill_single_tile_direct_formula():
    # With one tile the running max is the row max: o = sum q8(p) v / sum p.
    rng = np.random.default_rng(22)
    T, D = 100, 8
    K = [_bf16(rng.standard_normal((T, 1, D)))]
    V = [_bf16(rng.standard_normal((T, 1, D)))]
    q = _bf16(rng.standard_normal((1, 1, D)))
    one = np.ones(1, np.float32)
    out = attention.prefill_attention(q, [0, 1], K, V, one, one, one, block_n=128)
    Kt = e4m3.decode(e4m3.quantize(K[0][:, 0], 1.0))
    Vt = e4m3.decode(e4m3.quantize(V[0][:, 0], 1.0))
    qt = e4m3.decode(e4m3.quantize(q[0, 0], 1.0))
    s = Kt @ qt / math.sqrt(D)
    p = np.exp(s - s.max())
    pq = np.array([e4m3.decode(e4m3.encode(np.float32(np.float32(x) * np.float32(448.0))))[()] for x in p]) / 448
    np.testing.assert_allclose(out[0, 0], (pq @ Vt) / p.sum(), rtol=1e-12)


def test_prefill_tail_rows_equal_decode():
    # The last chunk row sits at position T-1 and sees the whole context: without P
    # rounding it equals decode attention over T keys; the first row equals decode over
    # T - Lq + 1 keys.
    rng = np.random.default_rng(23)
    T, Lq, Hq, Hkv, D = 90, 17, 4, 2, 8
    K = [_bf16(rng.standard_normal((T, Hkv, D)))]
    V = [_bf16(rng.standard_normal((T, Hkv, D)))]
    q = _bf16(rng.standard_normal((Lq, Hq, D)))
    s = np.float32(0.5)
    pre = attention.prefill_attention(q, [0, Lq], K, V, s, s, s, block_n=32, p_quant=False)
    for row, ctx in ((Lq - 1, T), (0, T - Lq + 1)):
        dec = attention.decode_attention_contiguous(q[row], K[0][:ctx], V[0][:ctx], s, s, s)
        for h in range(Hq):
            np.testing.assert_allclose(pre[row, h], dec[h], rtol=1e-12, atol=1e-13)


def test_prefill_window_matches_banded_sdpa_and_decode():
    # R6: with window W, the row at position p sees keys [p - W + 1, p]
    rng = np.random.default_rng(24)
    Hq, Hkv, D, W = 4, 2, 16, 37
    T, Lq = 150, 60
    K = [_bf16(rng.standard_normal((T, Hkv, D)))]
    V = [_bf16(rng.standard_normal((T, Hkv, D)))]
    q = _bf16(rng.standard_normal((Lq, Hq, D)))
    one = np.ones(1, np.float32)
    got = attention.prefill_attention(q, [0, Lq], K, V, one, one, one, block_n=32, fp8=False, window=W)
    qpos = T - Lq + np.arange(Lq)
    kpos = np.arange(T)
    mask = torch.from_numpy((kpos[None, :] <= qpos[:, None]) & (kpos[None, :] >= qpos[:, None] - W + 1))
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(K[0]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    vt = torch.from_numpy(V[0]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)
    # the last row equals decode over the last W keys (fp8, unrounded P)
    pre = attention.prefill_attention(q, [0, Lq], K, V, one, one, one, block_n=32, p_quant=False, window=W)
    dec = attention.decode_attention_contiguous(q[Lq - 1], K[0], V[0], one, one, one, window=W)
    for h in range(Hq):
        np.testing.assert_allclose(pre[Lq - 1, h], dec[h], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- split-K decode (R23)

def _dequant(K, V, qv_raw, qs, ks, vs):
    K8 = e4m3.decode(e4m3.quantize(K, ks)) * ks
    V8 = e4m3.decode(e4m3.quantize(V, vs)) * vs
    qv = e4m3.decode(e4m3.quantize(qv_raw, qs)) * qs
    return qv, K8, V8


@pytest.mark.parametrize("split_blocks", [1, 2, 3, 8])
@pytest.mark.parametrize("window", [0, 37])
def test_split_decode_with_exact_p_is_sdpa(split_blocks, window):
    """With exact P, splitting the keys and merging (acc, m, l) is the plain softmax:
    float64 scaled_dot_product_attention over the dequantised window."""
    rng = np.random.default_rng(20 + split_blocks + window)
    D, T = 8, 150
    lo = max(0, T - window) if window else 0
    qv, K, V = _dequant(rng.standard_normal((T, D)) * 2, rng.standard_normal((T, D)), rng.standard_normal(D),
                        np.float32(0.5), np.float32(0.75), np.float32(0.25))
    tau = 1 / math.sqrt(D)
    got = attention.split_decode(qv, K[lo:], V[lo:], T, lo, tau, split_blocks=split_blocks, block_n=32,
                                 p_quant=False, block_size=16)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qv)[None, None], torch.from_numpy(K[lo:])[None], torch.from_numpy(V[lo:])[None],
        scale=tau)[0, 0].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def _closed_form_fp8p(qv, K, V, T, lo, tau, split_blocks, block_n, bs):
    """Non-iterative statement of the split-K decode with FP8 P: key j of split s, tile t
    (tiles counted from the split's first block) gets the P code of e^(s_j - m) with m the
    maximum over the split's keys up to the end of tile t, and the weight
    dec(code) / 448 * e^(m - M); the denominator is sum_j e^(s_j - M), M the global max."""
    kpos = np.arange(lo, T)
    s = (K @ qv) * tau
    M = s.max()
    blk0 = lo // bs
    w = np.zeros(len(kpos))
    for j, kp in enumerate(kpos):
        split = (kp // bs - blk0) // split_blocks
        origin = (blk0 + split * split_blocks) * bs
        split_end = min((blk0 + (split + 1) * split_blocks) * bs, T)
        tile_end = min(origin + ((kp - origin) // block_n + 1) * block_n, split_end)
        m_run = s[(kpos >= max(origin, lo)) & (kpos < tile_end)].max()
        code = e4m3.encode(e4m3.fl32(e4m3.fl32(np.exp(s[j] - m_run)) * 448.0))
        w[j] = e4m3.decode(code) / 448.0 * math.exp(m_run - M)
    return (w @ V) / np.exp(s - M).sum()


@pytest.mark.parametrize("T,window,split_blocks,block_n", [
    (20, 0, 4, 32),      # one split, one partial tile: the single-tile direct formula
    (150, 0, 4, 32),     # splits of two 32-key tiles
    (150, 0, 3, 32),     # a split of 48 keys: a full tile and a partial one
    (300, 70, 2, 16),    # window starting inside block 14: split origins not tile-aligned
    (300, 200, 5, 32),   # window, splits of 80 keys (2.5 tiles)
    (257, 0, 16, 128),   # the kernel's shape: 128-key tiles, 256-key splits, a 1-key tail
])
def test_split_decode_fp8p_matches_closed_form(T, window, split_blocks, block_n):
    rng = np.random.default_rng(T + window + split_blocks)
    D = 8
    lo = max(0, T - window) if window else 0
    # strongly varying scores so that running maxima move between tiles and splits
    qv, K, V = _dequant(rng.standard_normal((T, D)) * 3, rng.standard_normal((T, D)), rng.standard_normal(D) * 2,
                        np.float32(0.5), np.float32(1.0), np.float32(0.25))
    tau = 1 / math.sqrt(D)
    got = attention.split_decode(qv, K[lo:], V[lo:], T, lo, tau, split_blocks=split_blocks, block_n=block_n,
                                 p_quant=True, block_size=16)
    ref = _closed_form_fp8p(qv, K[lo:], V[lo:], T, lo, tau, split_blocks, block_n, 16)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
    # the rounding is visible: exact P differs by more than rounding noise
    exact = attention.split_decode(qv, K[lo:], V[lo:], T, lo, tau, split_blocks=split_blocks, block_n=block_n,
                                   p_quant=False, block_size=16)
    assert np.abs(got - exact).max() > 1e-6


def test_split_decode_fp8p_depends_on_the_tile_origin():
    """Tiles start at each split's first block, not at absolute multiples of block_n: with
    a window the two readings give different P codes, and the oracle follows the first."""
    rng = np.random.default_rng(3)
    D, T, window = 8, 300, 180
    lo = T - window              # 120: the first split starts at key 112, 16 past a multiple of 32
    q = rng.standard_normal(D)
    # scores that rise along the keys, so that the running maximum moves in almost every tile
    K = rng.standard_normal((T, D)) + np.outer(np.arange(T) / 20.0, q / np.linalg.norm(q))
    qv, K, V = _dequant(K, rng.standard_normal((T, D)), q, np.float32(0.5), np.float32(1.0), np.float32(0.25))
    tau = 1 / math.sqrt(D)
    got = attention.split_decode(qv, K[lo:], V[lo:], T, lo, tau, split_blocks=64, block_n=32, p_quant=True)
    # absolute tiles: one tile walk over the window with tile0 = 0
    acc, m, l = attention._tile_walk(qv[None], K[lo:], V[lo:], np.array([T - 1]), lo, 32, tau, True, state=True)
    absolute = acc[0] / l[0]
    assert np.abs(got - absolute).max() > 1e-6
    ref = _closed_form_fp8p(qv, K[lo:], V[lo:], T, lo, tau, 64, 32, 16)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_decode_attention_split_mode_is_the_split_walk():
    """The paged entry point routes through the split walk per (sequence, head)."""
    rng = np.random.default_rng(4)
    Hq, Hkv, D = 4, 2, 8
    T_list = [1, 40, 150]
    q = _bf16(rng.standard_normal((len(T_list), Hq, D)) * 2)
    K = [_bf16(rng.standard_normal((t, Hkv, D)) * 3) for t in T_list]
    V = [_bf16(rng.standard_normal((t, Hkv, D))) for t in T_list]
    qs = np.array([0.5, 1.0, 0.25, 2.0], np.float32)
    ks = np.array([0.75, 0.125], np.float32)
    vs = np.array([1.5, 0.5], np.float32)
    kp, vp, table = _paged(K, V, T_list, rng, True, ks, vs)
    got = attention.decode_attention(q, kp, vp, table, T_list, qs, ks, vs, window=100, p_quant=True, split_blocks=2,
                                     block_n=16)
    tau = 1 / math.sqrt(D)
    for b, T in enumerate(T_list):
        lo = max(0, T - 100)
        for h in range(Hq):
            g = h // 2
            qv, K8, V8 = _dequant(K[b][:, g], V[b][:, g], q[b, h], qs[h], ks[g], vs[g])
            ref = _closed_form_fp8p(qv, K8[lo:], V8[lo:], T, lo, tau, 2, 16, 16)
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-12, atol=1e-13)


def test_e5m2_decode_matches_loops_and_sdpa():
    """An e5m2 layer (R25): the codes dequantised with their scales, the bf16 query, exact
    softmax — pure-Python loops with the e5m2 codec, and float64 SDPA."""
    from oracle import e5m2
    rng = np.random.default_rng(31)
    Hq, Hkv, D = 4, 2, 8
    T_list = [1, 9, 40]
    q = _bf16(rng.standard_normal((len(T_list), Hq, D)) * 2)
    K = [_bf16(rng.standard_normal((t, Hkv, D)) * 300) for t in T_list]
    V = [_bf16(rng.standard_normal((t, Hkv, D)) * 50) for t in T_list]
    ks = np.array([0.5, 2.0], np.float32)
    vs = np.array([0.25, 1.0], np.float32)
    one = np.ones(1, np.float32)
    B = len(T_list)
    nblk = [(t + BS - 1) // BS for t in T_list]
    table = np.full((B, max(nblk)), -1, np.int64)
    nb = sum(nblk)
    perm = rng.permutation(nb)
    off = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += nblk[b]
    kp = np.zeros((nb, Hkv, BS, D), np.uint8)
    vp = np.zeros((nb, Hkv, BS, D), np.uint8)
    for b in range(B):
        pos = np.arange(T_list[b])
        kvcache.cache_write(K[b], V[b], table[b, pos // BS] * BS + pos % BS, kp, vp, ks, vs, skip=False, fmt="e5m2")
    got = attention.decode_attention(q, kp, vp, table, T_list, one, ks, vs, fmt="e5m2")
    tau = 1 / math.sqrt(D)
    for b, T in enumerate(T_list):
        for h in range(Hq):
            g = h // 2
            Kd = [[float(e5m2.decode(e5m2.quantize(np.array([K[b][j][g][d]]), ks[g]))[0]) * float(ks[g])
                   for d in range(D)] for j in range(T)]
            Vd = [[float(e5m2.decode(e5m2.quantize(np.array([V[b][j][g][d]]), vs[g]))[0]) * float(vs[g])
                   for d in range(D)] for j in range(T)]
            sc = [sum(q[b, h, d] * Kd[j][d] for d in range(D)) * tau for j in range(T)]
            mx = max(sc)
            w = [math.exp(x - mx) for x in sc]
            z = sum(w)
            loop = [sum(w[j] * Vd[j][d] for j in range(T)) / z for d in range(D)]
            np.testing.assert_allclose(got[b, h], loop, rtol=1e-12, atol=1e-12)
            sd = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[b, h], dtype=torch.float64)[None, None], torch.tensor(Kd, dtype=torch.float64)[None],
                torch.tensor(Vd, dtype=torch.float64)[None], scale=tau)[0, 0]
            np.testing.assert_allclose(got[b, h], sd.numpy(), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- P-rounding error bound

def test_p_rounding_bound_exact_part_is_sdpa():
    rng = np.random.default_rng(40)
    D, T = 16, 90
    qv, K, V = _dequant(rng.standard_normal((T, D)) * 2, rng.standard_normal((T, D)), rng.standard_normal(D),
                        np.float32(0.5), np.float32(0.75), np.float32(0.25))
    tau = 1 / math.sqrt(D)
    o, B = attention.p_rounding_bound(qv, K, V, tau)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qv)[None, None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=tau)[0, 0]
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-13)
    assert np.all(B > 0)


@pytest.mark.parametrize("spread", [0.5, 3.0, 12.0])
@pytest.mark.parametrize("T,window,split_blocks,block_n", [
    (150, 0, 4, 32), (300, 70, 2, 16), (257, 0, 16, 128), (700, 0, 8, 128), (1000, 333, 1, 16)])
def test_split_decode_fp8p_within_the_p_rounding_bound(spread, T, window, split_blocks, block_n):
    """Every split and tile plan of the FP8-P decode stays within the bound: the score
    spreads reach p far below e4m3's normal range (subnormal codes and codes rounded to 0)."""
    rng = np.random.default_rng(int(spread * 10) + T + window + split_blocks)
    D = 8
    lo = max(0, T - window) if window else 0
    qv, K, V = _dequant(rng.standard_normal((T, D)) * spread, rng.standard_normal((T, D)),
                        rng.standard_normal(D) * 2, np.float32(0.5), np.float32(1.0), np.float32(0.25))
    tau = 1 / math.sqrt(D)
    got = attention.split_decode(qv, K[lo:], V[lo:], T, lo, tau, split_blocks=split_blocks, block_n=block_n,
                                 p_quant=True, block_size=16)
    o, B = attention.p_rounding_bound(qv, K[lo:], V[lo:], tau)
    assert np.all(np.abs(got - o) <= B * (1 + 1e-9))


def test_p_rounding_bound_is_reached_by_its_two_terms():
    """Two-key cases at the edges of the bound.  (a) p * 448 next to 4.25, a tie of e4m3
    between 4.0 and 4.5: the rounding error is 1/17 of p, 16/17 of the bound's 2^-4 p.
    (b) p * 448 just below 2^-10, half the smallest subnormal: the code is 0 and the
    error is the whole p, just below the bound's 2^-10 / 448."""
    tau = 1.0
    for p_target, lo_ratio in ((4.25 / 448.0, 0.93), (0.99 * 2.0 ** -10 / 448.0, 0.98)):
        K = np.array([[0.0], [math.log(p_target)]])
        qv = np.array([1.0])
        V = np.array([[0.0, 0.0], [1.0, 1.0]])
        got = attention.split_decode(qv, K, V, 2, 0, tau, split_blocks=1, block_n=16, p_quant=True, block_size=16)
        o, B = attention.p_rounding_bound(qv, K, V, tau)
        ratio = np.abs(got - o) / B
        assert np.all(ratio <= 1.0) and np.all(ratio >= lo_ratio), ratio
