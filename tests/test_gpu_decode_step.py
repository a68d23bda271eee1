"""fp8_decode_step on the GPU: the current token's cache write fused into the decode launch
must equal kv_quant_cache of that token followed by fp8_decode_attn — pool bytes and
output bit for bit.  The separate calls are pinned to the oracle by test_gpu_cache and
test_gpu_decode; equality carries that over.  Cases cover every head_dim, per-tensor and
per-head scales, windows, forced split counts, an empty sequence, and consecutive steps
whose current token opens a new pool block; the same on bf16 (skip) and e5m2 layers, whose
CUDA-core decode writes the current token in its launch too."""
import numpy as np
import pytest
import torch

import synth
from helpers import to_dev

f = pytest.importorskip("fp8_kv_cache_quant_gb300")
pytestmark = pytest.mark.gpu


def _scales(gran, q, k, v):
    if gran:
        return synth.amax_scales(q, 1), synth.amax_scales(k, 1), synth.amax_scales(v, 1)
    return torch.tensor([0.5]), torch.tensor([1.0]), torch.tensor([0.25])


def _kind_args(kind):
    """LayerCache.empty / call keywords of a layer kind: e4m3 pools, a skip layer's bf16
    pools, or e5m2 pools."""
    if kind == "bf16":
        return dict(bf16=True), dict(skip_layer_mask=[1])
    if kind == "e5m2":
        return dict(kv_format=f.KV_E5M2), {}
    return {}, {}


def _run_both(ctx, table, nb, q, k, v, qs, ks, vs, gran, window, splits, cache_a, cache_b, kind="e4m3"):
    """One decode step on two copies of a layer: (A) kv_quant_cache of the current token
    then fp8_decode_attn, (B) fp8_decode_step.  k / v hold every position of every
    sequence (sequence-major); the current token of sequence b is position ctx[b] - 1."""
    B = len(ctx)
    Hkv, D = k.shape[1], k.shape[2]
    cu = np.concatenate([[0], np.cumsum(ctx)])
    k_new = torch.zeros((B, Hkv, D), dtype=torch.bfloat16)
    v_new = torch.zeros((B, Hkv, D), dtype=torch.bfloat16)
    slots = np.full(B, -1, np.int64)
    all_slots = synth.slot_mapping(table, ctx)
    for b in range(B):
        if ctx[b] > 0:
            k_new[b] = k[cu[b + 1] - 1]
            v_new[b] = v[cu[b + 1] - 1]
            slots[b] = all_slots[cu[b + 1] - 1]
    _, kw = _kind_args(kind)
    args = (to_dev(table), to_dev(ctx), to_dev(qs), to_dev(ks), to_dev(vs), gran)
    f.kv_quant_cache(k_new.cuda(), v_new.cuda(), to_dev(slots), cache_a, to_dev(ks), to_dev(vs), gran, **kw)
    out_a = f.fp8_decode_attn(q.cuda(), cache_a, *args, window=window, num_splits=splits, **kw)
    out_b = f.fp8_decode_step(k_new.cuda(), v_new.cuda(), q.cuda(), cache_b, *args, window=window,
                              num_splits=splits, **kw)
    torch.cuda.synchronize()
    return out_a, out_b


def _layer_before_step(ctx, table, nb, k, v, ks, vs, gran, kind="e4m3"):
    """Two identical pools holding every position except each sequence's current token
    (stale bytes elsewhere are NaN codes, 0xFF)."""
    Hkv, D = k.shape[1], k.shape[2]
    cu = np.concatenate([[0], np.cumsum(ctx)])
    slots = synth.slot_mapping(table, ctx).copy()
    for b in range(len(ctx)):
        if ctx[b] > 0:
            slots[cu[b + 1] - 1] = -1
    ck, kw = _kind_args(kind)
    a = f.LayerCache.empty(nb, Hkv, D, **ck)
    a.k_cache.view(torch.uint8).fill_(0xFF)
    a.v_cache.view(torch.uint8).fill_(0xFF)
    if len(slots):
        f.kv_quant_cache(k.cuda(), v.cuda(), to_dev(slots), a, to_dev(ks), to_dev(vs), gran, **kw)
    b_ = f.LayerCache.empty(nb, Hkv, D, **ck)
    b_.k_cache.copy_(a.k_cache)
    b_.v_cache.copy_(a.v_cache)
    return a, b_


@pytest.mark.parametrize("D,G,gran,window,splits", [
    (128, 4, 1, 0, 0), (64, 8, 0, 0, 3), (256, 2, 1, 0, 0), (128, 16, 0, 50, 0), (64, 4, 1, 40, 2),
    (128, 1, 0, 0, 1), (256, 8, 0, 33, 0),
])
def test_decode_step_equals_write_then_decode(D, G, gran, window, splits):
    rng = np.random.default_rng(D * 5 + G + window + splits)
    Hkv = 2
    Hq = Hkv * G
    ctx = np.array([1, 15, 16, 17, 300, 1000, 0, 129], np.int32)
    table, nb = synth.block_table(ctx, seed=19, extra_blocks=2)
    n = int(ctx.sum())
    q = torch.from_numpy(rng.standard_normal((len(ctx), Hq, D)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy((rng.standard_normal((n, Hkv, D)) * 3.0).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    qs, ks, vs = _scales(gran, q, k, v)
    cache_a, cache_b = _layer_before_step(ctx, table, nb, k, v, ks.numpy(), vs.numpy(), gran)
    out_a, out_b = _run_both(ctx, table, nb, q, k, v, qs, ks, vs, gran, window, splits, cache_a, cache_b)
    assert torch.equal(cache_a.k_cache, cache_b.k_cache), "K pool differs"
    assert torch.equal(cache_a.v_cache, cache_b.v_cache), "V pool differs"
    assert torch.equal(out_a, out_b), "output differs"
    assert torch.all(out_b[6] == 0), "a sequence without keys gets a zero row"


def test_decode_step_consecutive_steps_across_a_block_boundary():
    """Three steps of a growing context through fp8_decode_step on one pool, against the
    separate calls on another: the current token moves from slot 14 to slot 0 of a new
    block (and in the long sequence past a split boundary)."""
    rng = np.random.default_rng(7)
    D, G, Hkv = 128, 4, 2
    Hq = Hkv * G
    final = np.array([17, 33, 3, 1666], np.int32)
    table, nb = synth.block_table(final, seed=23, extra_blocks=1)
    n = int(final.sum())
    k = torch.from_numpy((rng.standard_normal((n, Hkv, D)) * 2.0).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    ks, vs = synth.amax_scales(k, 1), synth.amax_scales(v, 1)
    qs = torch.full((Hq,), 0.05)
    cuf = np.concatenate([[0], np.cumsum(final)])
    start = final - 3  # the first step's context lengths (sequence 2 starts empty)

    def prefix(x, ctx):  # positions [0, ctx[b]) of every sequence, sequence-major
        return torch.cat([x[cuf[b]:cuf[b] + ctx[b]] for b in range(len(final))])

    cache_a, cache_b = _layer_before_step(start, table, nb, prefix(k, start), prefix(v, start), ks.numpy(),
                                          vs.numpy(), 1)
    for step in range(3):
        ctx = (start + step).astype(np.int32)
        kc, vc = prefix(k, ctx), prefix(v, ctx)
        q = torch.from_numpy(rng.standard_normal((len(final), Hq, D)).astype(np.float32)).to(torch.bfloat16)
        out_a, out_b = _run_both(ctx, table, nb, q, kc, vc, qs, ks, vs, 1, 0, 0, cache_a, cache_b)
        assert torch.equal(cache_a.k_cache, cache_b.k_cache), f"K pool differs at step {step}"
        assert torch.equal(cache_a.v_cache, cache_b.v_cache), f"V pool differs at step {step}"
        assert torch.equal(out_a, out_b), f"output differs at step {step}"


@pytest.mark.parametrize("kind,D,G,gran,window,splits", [
    ("bf16", 128, 4, 0, 0, 0), ("bf16", 64, 8, 0, 128, 0), ("bf16", 256, 2, 0, 0, 3), ("bf16", 64, 16, 0, 0, 2),
    ("e5m2", 128, 4, 1, 0, 0), ("e5m2", 64, 8, 0, 40, 2), ("e5m2", 256, 1, 1, 0, 0),
])
def test_decode_step_on_bf16_and_e5m2_layers(kind, D, G, gran, window, splits):
    """The CUDA-core decode's fused write: a skip layer's bf16 pools (an exact copy of the
    current token) and e5m2 pools (e5m2 of x / s) — the same bytes and output as
    kv_quant_cache then fp8_decode_attn, so a bf16 decode step compares with the e4m3 one
    launch for launch."""
    rng = np.random.default_rng(D * 3 + G + window + splits + (kind == "e5m2"))
    Hkv = 2
    Hq = Hkv * G
    ctx = np.array([1, 15, 16, 17, 300, 1000, 0, 129], np.int32)
    table, nb = synth.block_table(ctx, seed=29, extra_blocks=2)
    n = int(ctx.sum())
    q = torch.from_numpy(rng.standard_normal((len(ctx), Hq, D)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy((rng.standard_normal((n, Hkv, D)) * 3.0).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    qs, ks, vs = _scales(gran, q, k, v)
    if kind == "e5m2":
        ks, vs = ks * 0.01, vs * 0.01   # scaled values far past e4m3's range, inside e5m2's
    cache_a, cache_b = _layer_before_step(ctx, table, nb, k, v, ks.numpy(), vs.numpy(), gran, kind)
    out_a, out_b = _run_both(ctx, table, nb, q, k, v, qs, ks, vs, gran, window, splits, cache_a, cache_b, kind)
    # bit patterns: stale slots hold NaN codes, which never compare equal as values
    bits = lambda t: t.view(torch.uint8)
    assert torch.equal(bits(cache_a.k_cache), bits(cache_b.k_cache)), "K pool differs"
    assert torch.equal(bits(cache_a.v_cache), bits(cache_b.v_cache)), "V pool differs"
    assert torch.equal(out_a, out_b), "output differs"
    assert torch.isfinite(out_b.float()).all()
    assert torch.all(out_b[6] == 0), "a sequence without keys gets a zero row"


def test_decode_step_oversized_context_writes_nothing():
    """A context length beyond what the block table can address is clamped and reported
    (FKV_FAULT_CONTEXT); the fused write must then leave every pool byte as it was,
    since position T - 1 of the clamped range is one of the caller's cached tokens."""
    rng = np.random.default_rng(17)
    ctx = np.array([40, 20], np.int32)
    table, nb = synth.block_table(ctx, seed=2)
    Hkv, D, Hq = 2, 128, 8
    n = int(ctx.sum())
    k = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    q = torch.from_numpy(rng.standard_normal((2, Hq, D)).astype(np.float32)).to(torch.bfloat16)
    one = torch.ones(1)
    cache = f.LayerCache.empty(nb, Hkv, D)
    cache.k_cache.zero_()
    cache.v_cache.zero_()
    f.kv_quant_cache(k.cuda(), v.cuda(), to_dev(synth.slot_mapping(table, ctx)), cache, to_dev(one), to_dev(one), 0)
    k_before, v_before = cache.k_cache.clone(), cache.v_cache.clone()
    k_new = torch.full((2, Hkv, D), 3.0, dtype=torch.bfloat16)
    v_new = torch.full((2, Hkv, D), -3.0, dtype=torch.bfloat16)
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    long_ctx = np.array([10_000, -5], np.int32)   # beyond the table's 3 blocks; negative
    o = f.fp8_decode_step(k_new.cuda(), v_new.cuda(), q.cuda(), cache, to_dev(table), to_dev(long_ctx),
                          to_dev(one), to_dev(one), to_dev(one), 0, fault=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) & f.FAULT_CONTEXT
    assert torch.isfinite(o.float()).all()
    assert torch.equal(cache.k_cache, k_before) and torch.equal(cache.v_cache, v_before)
