"""kv_quant_cache on the GPU against the oracle: cache bytes must match bit-exactly."""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_pools, to_dev
from oracle import e4m3, kvcache

f = pytest.importorskip("fp8_kv_cache_quant_gb300")
pytestmark = pytest.mark.gpu


def _all_bf16_patterns(D=128):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    n = 65536 // D
    return torch.from_numpy(bits.view(np.int16).reshape(n, 1, D).copy()).view(torch.bfloat16)


@pytest.mark.parametrize("scale", [1.0, 0.0371, 3.5])
def test_codec_every_bf16_pattern(scale):
    """Every bf16 bit pattern (NaN and +-inf included) through the e4m3 cache write."""
    k = _all_bf16_patterns()
    v = k.flip(0).contiguous()
    n, H, D = k.shape
    cache = f.LayerCache.empty(n // 16, H, D)
    slots = torch.arange(n, dtype=torch.int64, device="cuda")
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    f.kv_quant_cache(k.cuda(), v.cuda(), slots, cache, s, s, f.SCALE_PER_TENSOR)
    got_k = cache.k_cache.cpu().numpy().reshape(n, D)
    got_v = cache.v_cache.cpu().numpy().reshape(n, D)
    ref_k = e4m3.quantize(synth.bf16_to_f64(k).reshape(n, D), np.float32(scale))
    ref_v = e4m3.quantize(synth.bf16_to_f64(v).reshape(n, D), np.float32(scale))
    assert np.array_equal(got_k, ref_k)
    assert np.array_equal(got_v, ref_v)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("gran", [0, 1])
def test_cache_write_per_head_scales_sentinel(D, gran):
    rng = np.random.default_rng(D + gran)
    H = 4
    ctx = np.array([1, 17, 50, 3], np.int32)
    table, nb = synth.block_table(ctx, seed=7, extra_blocks=5)
    n = int(ctx.sum())
    k = torch.from_numpy((rng.standard_normal((n, H, D)) * 5).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, H, D)).astype(np.float32)).to(torch.bfloat16)
    if gran:
        ks = synth.amax_scales(k, 1).numpy()
        vs = synth.amax_scales(v, 1).numpy()
    else:
        ks = np.array([0.75], np.float32)
        vs = np.array([0.02], np.float32)
    slots = synth.slot_mapping(table, ctx)
    slots[5] = -1  # padding token: skipped
    cache = f.LayerCache.empty(nb, H, D)
    cache.k_cache.fill_(0xA5)
    cache.v_cache.fill_(0x5A)
    f.kv_quant_cache(k.cuda(), v.cuda(), to_dev(slots), cache, to_dev(ks), to_dev(vs), gran)
    kp = np.full((nb, H, 16, D), 0xA5, np.uint8)
    vp = np.full((nb, H, 16, D), 0x5A, np.uint8)
    kvcache.cache_write(synth.bf16_to_f64(k), synth.bf16_to_f64(v), slots, kp, vp, ks, vs, skip=False)
    assert np.array_equal(cache.k_cache.cpu().numpy(), kp)
    assert np.array_equal(cache.v_cache.cpu().numpy(), vp)


def test_skip_layer_exact_bf16_copy():
    rng = np.random.default_rng(5)
    ctx = np.array([33, 7], np.int32)
    table, nb = synth.block_table(ctx, seed=3)
    n, H, D = int(ctx.sum()), 2, 64
    k = torch.from_numpy(rng.standard_normal((n, H, D)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, H, D)).astype(np.float32)).to(torch.bfloat16)
    cache = f.LayerCache.empty(nb, H, D, bf16=True)
    cache.k_cache.zero_()
    cache.v_cache.zero_()
    mask = np.array([0, 1, 0], np.uint8)
    f.kv_quant_cache(k.cuda(), v.cuda(), to_dev(synth.slot_mapping(table, ctx)), cache, None, None, 0,
                     layer=1, skip_layer_mask=mask)
    kp, vp = oracle_pools(kvcache, ctx, table, nb, k, v, [1.0], [1.0], bf16_layer=True)
    assert np.array_equal(cache.k_cache.float().cpu().numpy(), kp)
    assert np.array_equal(cache.v_cache.float().cpu().numpy(), vp)


def test_slot_out_of_range_raises_fault_and_writes_nothing():
    H, D = 1, 64
    cache = f.LayerCache.empty(2, H, D)
    cache.k_cache.fill_(7)
    cache.v_cache.fill_(7)
    k = torch.ones((2, H, D), dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([32, 1000], dtype=torch.int64, device="cuda")   # capacity is 32 slots
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    one = torch.ones(1, device="cuda")
    f.kv_quant_cache(k, k, slots, cache, one, one, 0, fault=fault)
    assert int(fault.item()) & f.FAULT_SLOT
    assert torch.all(cache.k_cache == 7) and torch.all(cache.v_cache == 7)


def test_prefill_workload_fill_sampled_blocks():
    """Full-size fill of the head_dim-256 prefill workload (4 x 32768 tokens), sampled
    blocks compared bit-exactly with the oracle's quantisation."""
    w = synth.WORKLOADS[5]
    data = synth.prefill_data(w, device="cuda")
    ctx = np.full(w.batch, w.seq_len, np.int32)
    table, nb = synth.block_table(ctx, seed=w.seed)
    cache = f.LayerCache.empty(nb, w.num_kv_heads, w.head_dim)
    f.kv_quant_cache(data.k, data.v, to_dev(synth.slot_mapping(table, ctx)), cache, data.k_scale, data.v_scale,
                     f.SCALE_PER_HEAD)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    ks, vs = data.k_scale.cpu().numpy(), data.v_scale.cpu().numpy()
    for b in range(w.batch):
        for lb in list(rng.choice(w.seq_len // 16, 6, replace=False)) + [0, w.seq_len // 16 - 1]:
            pb = table[b, lb]
            rows = slice(b * w.seq_len + lb * 16, b * w.seq_len + lb * 16 + 16)
            kx = synth.bf16_to_f64(data.k[rows])       # [16][1][D]
            vx = synth.bf16_to_f64(data.v[rows])
            got_k = cache.k_cache[pb, 0].cpu().numpy()
            got_v = cache.v_cache[pb, 0].cpu().numpy()
            assert np.array_equal(got_k, e4m3.quantize(kx[:, 0], ks[0]))
            assert np.array_equal(got_v, e4m3.quantize(vx[:, 0], vs[0]))


@pytest.mark.parametrize("scale", [1.0, 0.0371])
def test_clip_counts_every_bf16_pattern(scale):
    """The counting cache write over every bf16 bit pattern: the counts equal the oracle's
    (integers, exact) and the cache bytes equal those of the plain write."""
    k = _all_bf16_patterns()
    v = k.flip(0).contiguous()
    n, H, D = k.shape
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    slots = torch.arange(n, dtype=torch.int64, device="cuda")
    plain = f.LayerCache.empty(n // 16, H, D)
    f.kv_quant_cache(k.cuda(), v.cuda(), slots, plain, s, s, f.SCALE_PER_TENSOR)
    counted = f.LayerCache.empty(n // 16, H, D)
    counts = f.kv_quant_cache_clips(k.cuda(), v.cuda(), slots, counted, s, s, f.SCALE_PER_TENSOR)
    torch.cuda.synchronize()
    assert torch.equal(plain.k_cache, counted.k_cache) and torch.equal(plain.v_cache, counted.v_cache)
    got = counts.cpu().tolist()
    ref = [kvcache.clip_count(synth.bf16_to_f64(k), np.float32(scale)),
           kvcache.clip_count(synth.bf16_to_f64(v), np.float32(scale))]
    assert got == ref and ref[0] > 0


def test_clip_counts_per_head_accumulate_and_skip_layers():
    """Per-head scales with planted outliers; two calls accumulate; a skip layer clips nothing."""
    rng = np.random.default_rng(12)
    n, H, D = 300, 4, 128
    k = torch.from_numpy((rng.standard_normal((n, H, D)) * 40).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy((rng.standard_normal((n, H, D)) * 40).astype(np.float32)).to(torch.bfloat16)
    k[5, 1, 7] = 30000.0
    v[77, 3, 0] = -9000.0
    ks = np.array([0.2, 0.5, 0.1, 1.0], np.float32)
    vs = np.array([0.3, 0.05, 0.25, 0.5], np.float32)
    ctx = np.array([n], np.int32)
    table, nb = synth.block_table(ctx, seed=2)
    slots = to_dev(synth.slot_mapping(table, ctx))
    cache = f.LayerCache.empty(nb, H, D)
    counts = f.kv_quant_cache_clips(k.cuda(), v.cuda(), slots, cache, to_dev(ks), to_dev(vs), f.SCALE_PER_HEAD)
    counts = f.kv_quant_cache_clips(k.cuda(), v.cuda(), slots, cache, to_dev(ks), to_dev(vs), f.SCALE_PER_HEAD,
                                    clip_counts=counts)
    ref = [kvcache.clip_count(synth.bf16_to_f64(k), ks), kvcache.clip_count(synth.bf16_to_f64(v), vs)]
    assert counts.cpu().tolist() == [2 * ref[0], 2 * ref[1]] and ref[0] > 1 and ref[1] > 1
    bf = f.LayerCache.empty(nb, H, D, bf16=True)
    c2 = f.kv_quant_cache_clips(k.cuda(), v.cuda(), slots, bf, None, None, f.SCALE_PER_TENSOR, skip_layer_mask=[1])
    assert c2.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("scale", [1.0, 0.0371, 3.5])
def test_e5m2_codec_every_bf16_pattern(scale):
    """Every bf16 bit pattern through the e5m2 cache write (pools with kv_format KV_E5M2),
    bit-exact against the oracle's e5m2 codec, with the clip counts at the e5m2 limit."""
    from oracle import e5m2
    k = _all_bf16_patterns()
    v = k.flip(0).contiguous()
    n, H, D = k.shape
    cache = f.LayerCache.empty(n // 16, H, D, kv_format=f.KV_E5M2)
    slots = torch.arange(n, dtype=torch.int64, device="cuda")
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    counts = f.kv_quant_cache_clips(k.cuda(), v.cuda(), slots, cache, s, s, f.SCALE_PER_TENSOR)
    got_k = cache.k_cache.cpu().numpy().reshape(n, D)
    got_v = cache.v_cache.cpu().numpy().reshape(n, D)
    kx, vx = synth.bf16_to_f64(k), synth.bf16_to_f64(v)
    assert np.array_equal(got_k, e5m2.quantize(kx.reshape(n, D), np.float32(scale)))
    assert np.array_equal(got_v, e5m2.quantize(vx.reshape(n, D), np.float32(scale)))
    assert counts.cpu().tolist() == [kvcache.clip_count(kx, np.float32(scale), limit=e5m2.E5M2_MAX),
                                     kvcache.clip_count(vx, np.float32(scale), limit=e5m2.E5M2_MAX)]
