"""Pins of the oracle's paged cache write and the KV memory formula (CPU only)."""
import numpy as np
import torch

import synth
from oracle import e4m3, kvcache


def test_cache_write_lands_at_slot_and_nowhere_else():
    rng = np.random.default_rng(30)
    nb, H, bs, D = 7, 3, 16, 8
    kp = np.full((nb, H, bs, D), 0xA5, np.uint8)
    vp = np.full((nb, H, bs, D), 0x5A, np.uint8)
    k = rng.standard_normal((5, H, D)) * 4
    v = rng.standard_normal((5, H, D))
    slots = np.array([3, 17, -1, 111, 64])
    ks = np.array([0.5, 1.0, 2.0], np.float32)
    vs = np.array([0.25], np.float32)
    kvcache.cache_write(k, v, slots, kp, vp, ks, vs, skip=False)
    touched = np.zeros((nb, H, bs), bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        touched[s // bs, :, s % bs] = True
        for h in range(H):
            # head h uses its own K scale, the single V scale for every head
            assert np.array_equal(kp[s // bs, h, s % bs], e4m3.quantize(k[t, h], ks[h]))
            assert np.array_equal(vp[s // bs, h, s % bs], e4m3.quantize(v[t, h], vs[0]))
    assert np.all(kp[~touched] == 0xA5) and np.all(vp[~touched] == 0x5A)


def test_skip_layer_is_exact_bf16_copy():
    rng = np.random.default_rng(31)
    x = torch.from_numpy(rng.standard_normal((4, 2, 8)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    kp = np.zeros((2, 2, 16, 8), np.uint16)
    vp = np.zeros((2, 2, 16, 8), np.uint16)
    kvcache.cache_write(bits, bits, np.array([0, 5, 16, 31]), kp, vp, None, None, skip=True)
    assert np.array_equal(kp[1, :, 15], bits[3])
    assert np.array_equal(vp[0, :, 5], bits[1])


def test_memory_formula_matches_pool_bytes():
    # M_KV = 2 L H_KV D T B S for block-aligned T; the paged pool adds the block remainder.
    L, H, D = 4, 8, 128
    T = [4096] * 3
    assert kvcache.paged_kv_bytes(H, D, T, [1] * L) == kvcache.kv_bytes_formula(L, H, D, 4096, 3, 1)
    ctx = synth.context_lengths(8, 16384, 24576, seed=1)
    table, nb = synth.block_table(ctx, seed=1)
    pool_bytes_one_layer_fp8 = 2 * nb * H * 16 * D * 1           # k and v pools as allocated
    assert kvcache.paged_kv_bytes(H, D, ctx, [1]) == pool_bytes_one_layer_fp8
    # mixed bf16 / e4m3 layers (the skip-layer mask) are counted per layer
    mixed = kvcache.paged_kv_bytes(H, D, ctx, [1, 2, 1, 2])
    assert mixed == 2 * pool_bytes_one_layer_fp8 + 2 * 2 * pool_bytes_one_layer_fp8
    # the formula's value is never above the paged allocation and the remainder < one block
    tok = int(np.sum(ctx))
    exact = 2 * H * D * tok
    assert 0 <= pool_bytes_one_layer_fp8 - exact < 2 * H * D * 16 * len(ctx)


def test_clip_count_hand_values():
    """Scale 1: 448 is representable (kept); 450, -450, +-inf are clipped; NaN is not a
    clip.  Scale 0.5 doubles the values: 224 -> 448 (kept), 226 -> 452 (clipped)."""
    x = np.array([448.0, 450.0, -450.0, 416.0, np.inf, -np.inf, np.nan, 0.0]).reshape(1, 1, -1)
    assert kvcache.clip_count(x, np.float32(1.0)) == 4
    y = np.array([224.0, 226.0, -226.0, 100.0]).reshape(1, 1, -1)
    assert kvcache.clip_count(y, np.float32(0.5)) == 2
    # one scale per head (axis 1): head 0 at scale 1 keeps 300, head 1 at scale 0.5 clips it
    z = np.array([[[300.0, 10.0], [300.0, 10.0]]])
    assert kvcache.clip_count(z, np.array([1.0, 0.5], np.float32)) == 1


def test_clip_count_matches_float32_arithmetic_and_the_codec():
    """Brute force with numpy float32 arithmetic (IEEE single multiply by the single
    reciprocal), element by element; every clipped element encodes to +-448."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 3, 16)) * 120.0
    x[0, 1, 3] = 2000.0
    x[4, 2, 0] = -7000.0
    x = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
    s = np.array([0.75, 0.3, 1.25], np.float32)
    n = 0
    for idx in np.ndindex(*x.shape):
        inv = np.float32(1.0) / s[idx[1]]
        yv = np.float32(x[idx]) * inv
        if abs(float(yv)) > 448.0:
            n += 1
            code = int(e4m3.quantize(np.array([x[idx]]), s[idx[1]])[0])
            assert code in (0x7E, 0xFE)
    assert n > 2
    assert kvcache.clip_count(x, s) == n
