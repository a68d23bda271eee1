"""fp8_decode_attn (split-K paged decode + FP32 merge) on the GPU against the oracle.

Tolerance: max-abs 2e-2 and relative L2 1e-2 of the oracle's float64 FP8-emulated
result.  Where the library rounds P (the tensor-core decode of e4m3 layers), the oracle
walks the same splits and tiles with P rounded (reading R23); elsewhere P is exact and
the oracle is the plain softmax.  The split size the oracle walks is never asked of the
library: every test fixes the split count and derives the blocks per split from the rule
the header documents (restated in helpers.decode_split_blocks), and asserts that the
library reports the same; the automatic plan is checked on the benchmark's layer with a
split size derived by hand for a 152-SM GB300.  Every e4m3 result is also compared with
the plain softmax definition (P exact), within the element-wise bound that e4m3 rounding
of P allows (oracle.attention.p_rounding_bound); the distances are recorded as test
properties (rel_l2_vs_exact, worst_err_over_bound).
Small cases cover every head_dim, several GQA group sizes, both scale granularities, the
bf16 skip-layer path, windows, ragged and empty contexts and forced split counts; the
full-size workloads are checked on sampled sequences and heads with the split plan the
benchmark runs on a 152-SM GB300.
"""
import math

import numpy as np
import pytest
import torch

import synth
from helpers import (assert_close, assert_within_p_bound, auto_split_blocks, build_layer, decode_block_n,
                     decode_split_blocks, oracle_pools, to_dev)
from oracle import attention, e4m3, kvcache

f = pytest.importorskip("fp8_kv_cache_quant_gb300")
pytestmark = pytest.mark.gpu


def _oracle_mode(D, bf16_layer, batch, Hq, Hkv, max_blocks, window, num_splits):
    """Keyword arguments of the oracle's decode for the kernel the layer runs.  bf16 layers:
    P exact, the plain softmax.  e4m3 layers: P rounded per tile (128 keys, 256 at
    head_dim 64) of each split (R23), with the blocks per split of the documented rule
    for this split count."""
    if bf16_layer:
        assert f.fkv_decode_block_n(D, True) == 0
        return {}
    assert num_splits > 0, "e4m3 parity cases fix their split count"
    assert f.fkv_decode_block_n(D) == decode_block_n(D)
    bps = decode_split_blocks(max_blocks, window, num_splits, D)
    assert f.fp8_decode_attn_split_blocks(batch, Hq, Hkv, D, max_blocks, window, num_splits) == bps
    return dict(p_quant=True, split_blocks=bps, block_n=decode_block_n(D))


def _inputs(rng, ctx, Hq, Hkv, D, scale_k=3.0):
    n = int(np.sum(ctx))
    q = torch.from_numpy(rng.standard_normal((len(ctx), Hq, D)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy((rng.standard_normal((n, Hkv, D)) * scale_k).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    return q, k, v


CASES = [
    # D, G, bf16 layer, gran, window, num_splits (0: automatic, bf16 layers only)
    (128, 4, False, 0, 0, 4),
    (128, 4, False, 1, 0, 3),
    (64, 8, False, 1, 0, 2),
    (64, 8, True, 0, 128, 0),
    (128, 8, False, 0, 0, 1),
    (256, 1, False, 1, 0, 6),
    (256, 8, True, 0, 0, 2),
    (128, 16, False, 1, 50, 1),
    (64, 2, False, 0, 0, 5),
    (128, 1, True, 0, 0, 0),
    (64, 16, True, 1, 0, 0),
    (256, 4, False, 0, 33, 1),
    (64, 4, False, 1, 0, 8),
    (64, 4, False, 0, 77, 1),
    (64, 8, False, 1, 300, 2),
]


@pytest.mark.parametrize("D,G,bf16_layer,gran,window,splits", CASES)
def test_decode_small_parity(D, G, bf16_layer, gran, window, splits, record_property):
    rng = np.random.default_rng(D * 7 + G * 3 + window + splits)
    Hkv = 2
    Hq = Hkv * G
    ctx = np.array([1, 15, 16, 17, 300, 1000, 0, 129], np.int32)
    table, nb = synth.block_table(ctx, seed=11, extra_blocks=2)
    q, k, v = _inputs(rng, ctx, Hq, Hkv, D)
    if gran:
        qs, ks, vs = synth.amax_scales(q, 1), synth.amax_scales(k, 1), synth.amax_scales(v, 1)
    else:
        qs = torch.tensor([0.5]); ks = torch.tensor([1.0]); vs = torch.tensor([0.25])
    # stale bytes of partly filled blocks are NaN codes (0xFF): they must not leak into the result
    cache = build_layer(f, ctx, table, nb, k, v, ks.numpy(), vs.numpy(), gran, bf16_layer, sentinel=0xFF)
    mask = [1] if bf16_layer else None
    out = f.fp8_decode_attn(q.cuda(), cache, to_dev(table), to_dev(ctx), to_dev(qs), to_dev(ks), to_dev(vs),
                            gran, window=window, skip_layer_mask=mask, num_splits=splits)
    kp, vp = oracle_pools(kvcache, ctx, table, nb, k, v, ks.numpy(), vs.numpy(), bf16_layer)
    mode = _oracle_mode(D, bf16_layer, len(ctx), Hq, Hkv, table.shape[1], window, splits)
    ref = attention.decode_attention(synth.bf16_to_f64(q), kp, vp, table, ctx, qs.numpy(), ks.numpy(), vs.numpy(),
                                     fp8=not bf16_layer, window=window, **mode)
    got = out.float().cpu().numpy()
    assert np.all(got[6] == 0), "empty context must give a zero row"
    what = f"D={D} G={G} bf16={bf16_layer} gran={gran} W={window} splits={splits}"
    assert_close(got, ref, what=what)
    if not bf16_layer:
        exact, bound = attention.decode_attention(synth.bf16_to_f64(q), kp, vp, table, ctx, qs.numpy(), ks.numpy(),
                                                  vs.numpy(), window=window, p_bound=True)
        r, worst = assert_within_p_bound(got, exact, bound, what=what + " vs exact softmax")
        record_property("rel_l2_vs_exact", r)
        record_property("worst_err_over_bound", worst)


@pytest.mark.parametrize("D,G,gran,window,splits", [
    (128, 4, 1, 0, 0), (64, 8, 0, 0, 3), (256, 2, 1, 0, 0), (128, 16, 0, 100, 0), (64, 4, 1, 40, 2),
])
def test_decode_e5m2_layers(D, G, gran, window, splits):
    """e5m2 pools (kv_format KV_E5M2): the codes dequantised with their scales, the bf16
    query and exact P (R25) on the CUDA cores, against the oracle's e5m2 decode."""
    rng = np.random.default_rng(D + G + window)
    Hkv = 2
    Hq = Hkv * G
    ctx = np.array([1, 15, 16, 17, 300, 1000, 0, 129], np.int32)
    table, nb = synth.block_table(ctx, seed=13, extra_blocks=2)
    q, k, v = _inputs(rng, ctx, Hq, Hkv, D, scale_k=40.0)
    if gran:
        ks, vs = synth.amax_scales(k, 1) * (448.0 / 57344.0), synth.amax_scales(v, 1) * (448.0 / 57344.0)
    else:
        ks = torch.tensor([0.01]); vs = torch.tensor([0.002])
    qs = torch.ones(1)
    cache = build_layer(f, ctx, table, nb, k, v, ks.numpy(), vs.numpy(), gran, False, sentinel=0xFF,
                        kv_format=f.KV_E5M2)
    out = f.fp8_decode_attn(q.cuda(), cache, to_dev(table), to_dev(ctx), to_dev(qs), to_dev(ks), to_dev(vs), gran,
                            window=window, num_splits=splits)
    kp, vp = oracle_pools(kvcache, ctx, table, nb, k, v, ks.numpy(), vs.numpy(), False, fmt="e5m2")
    ref = attention.decode_attention(synth.bf16_to_f64(q), kp, vp, table, ctx, qs.numpy(), ks.numpy(), vs.numpy(),
                                     window=window, fmt="e5m2")
    got = out.float().cpu().numpy()
    assert np.all(got[6] == 0), "empty context must give a zero row"
    assert_close(got, ref, what=f"e5m2 D={D} G={G} gran={gran} W={window} splits={splits}")


@pytest.mark.parametrize("Hkv,G,D", [(3, 2, 64), (1, 8, 64), (5, 4, 64), (3, 4, 128)])
def test_decode_odd_kv_head_counts(Hkv, G, D):
    """Odd KV head counts and a single KV head, on both decode kernels."""
    rng = np.random.default_rng(Hkv * 10 + G)
    Hq = Hkv * G
    ctx = np.array([300, 1, 1000, 129], np.int32)
    table, nb = synth.block_table(ctx, seed=7, extra_blocks=2)
    q, k, v = _inputs(rng, ctx, Hq, Hkv, D)
    qs, ks, vs = synth.amax_scales(q, 1), synth.amax_scales(k, 1), synth.amax_scales(v, 1)
    cache = build_layer(f, ctx, table, nb, k, v, ks.numpy(), vs.numpy(), 1, False, sentinel=0xFF)
    out = f.fp8_decode_attn(q.cuda(), cache, to_dev(table), to_dev(ctx), to_dev(qs), to_dev(ks), to_dev(vs), 1,
                            num_splits=3)
    kp, vp = oracle_pools(kvcache, ctx, table, nb, k, v, ks.numpy(), vs.numpy(), False)
    mode = _oracle_mode(D, False, len(ctx), Hq, Hkv, table.shape[1], 0, 3)
    ref = attention.decode_attention(synth.bf16_to_f64(q), kp, vp, table, ctx, qs.numpy(), ks.numpy(), vs.numpy(),
                                     **mode)
    assert_close(out.float().cpu().numpy(), ref, what=f"Hkv={Hkv} G={G} D={D}")


@pytest.mark.parametrize("D", [128, 64])
def test_split_count_invariance_and_permutation(D):
    rng = np.random.default_rng(3)
    Hq, Hkv = 32, 8
    ctx = np.array([2000, 777, 4096], np.int32)
    table, nb = synth.block_table(ctx, seed=5)
    q, k, v = _inputs(rng, ctx, Hq, Hkv, D)
    one = np.ones(1, np.float32)
    cache = build_layer(f, ctx, table, nb, k, v, one, one, 0, False, sentinel=0xFF)
    outs = {}
    for s in (1, 2, 7, 0):
        outs[s] = f.fp8_decode_attn(q.cuda(), cache, to_dev(table), to_dev(ctx), to_dev(one), to_dev(one),
                                    to_dev(one), 0, num_splits=s).float().cpu().numpy()
    assert np.all(np.isfinite(outs[1]))
    if f.fkv_decode_block_n(D) > 0:
        # P rounded per split and tile: each split count against the oracle walking the
        # same splits (their P codes differ by design); the automatic plan's split size is
        # the documented rule evaluated for this device's SM count
        kp, vp = oracle_pools(kvcache, ctx, table, nb, k, v, one, one, False)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        for s, o in outs.items():
            if s > 0:
                mode = _oracle_mode(D, False, len(ctx), Hq, Hkv, table.shape[1], 0, s)
            else:
                bps = auto_split_blocks(len(ctx), Hkv, table.shape[1], 0, sms, D)
                assert f.fp8_decode_attn_split_blocks(len(ctx), Hq, Hkv, D, table.shape[1]) == bps
                mode = dict(p_quant=True, split_blocks=bps, block_n=decode_block_n(D))
            ref = attention.decode_attention(synth.bf16_to_f64(q), kp, vp, table, ctx, one, one, one, **mode)
            assert_close(o, ref, what=f"num_splits={s}")
    else:
        # exact P: different split counts group the keys differently; the per-tile f16
        # P.V partials then round differently, at about 1e-3 of the output's scale
        scale = float(np.max(np.abs(outs[1])))
        for s in (2, 7, 0):
            np.testing.assert_allclose(outs[s], outs[1], rtol=2.0 ** -7, atol=2e-3 * scale)
            assert np.linalg.norm(outs[s] - outs[1]) <= 2e-3 * np.linalg.norm(outs[1])
    # the same data under another physical block permutation: bit-identical output
    table2, nb2 = synth.block_table(ctx, seed=99, extra_blocks=3)
    cache2 = build_layer(f, ctx, table2, nb2, k, v, one, one, 0, False, sentinel=0x7F)
    o2 = f.fp8_decode_attn(q.cuda(), cache2, to_dev(table2), to_dev(ctx), to_dev(one), to_dev(one), to_dev(one), 0,
                           num_splits=7).float().cpu().numpy()
    assert np.array_equal(o2, outs[7])


# Split counts of the full-size workloads: the automatic plan of a 152-SM GB300 (456
# resident CTAs, 3 per SM), derived by hand from the documented rule (waves x blocks per
# split minimal, ties to the longer split), passed explicitly so that the tests do not
# depend on the SM count of the device they run on:
#   1: 8 units (1 sequence x 8 KV heads), 256 blocks: 8 blocks per split -> 32 splits,
#      256 CTAs, one wave of cost 8 (any longer split costs more) -> num_splits 32;
#   2: 64 units, 1,447 blocks: 208 -> 7 splits, 448 CTAs, one wave, cost 208 (104 would
#      take two waves, cost 208 too; the tie goes to 208) -> num_splits 7 (ceil(1447 / 7)
#      = 207 -> 208);
#   3: full layers 64 units, 1,774 blocks: 256 -> 7 splits, 448 CTAs, cost 256 (224 needs
#      8 splits, 512 CTAs, two waves) -> 7 (ceil(1774 / 7) = 254 -> 256); window-128
#      layers span at most 9 blocks: 8 -> 2 splits -> 2;
#   4: 8 units, 8,192 blocks: 144 -> 57 splits, 456 CTAs, exactly one wave (136 needs 61
#      splits, 488 CTAs) -> 57 (ceil(8192 / 57) = 144).
WORKLOAD_SPLITS = {1: {0: 32}, 2: {0: 7}, 3: {0: 7, 128: 1}, 4: {0: 57}}


def _decode_layer_check(w, layer, ctx, table, nb, seqs, heads, num_splits=None, exact=None, auto_bps=None):
    """Build one full-size layer through the C ABI and compare sampled (b, h) with the
    oracle computed from the contiguous bf16 inputs.  num_splits None: the workload's
    split count (WORKLOAD_SPLITS); 0: the automatic plan, whose blocks per split the
    caller gives as ``auto_bps``.  With a list ``exact`` (e4m3 layers) the plain softmax
    results and their P-rounding bounds of the same (b, h) are appended to it."""
    data = synth.decode_layer(w, layer, ctx, device="cuda")
    bf16_layer = bool(w.skip_mask()[layer])
    gran = f.SCALE_PER_HEAD if w.scale_mode == "amax" else f.SCALE_PER_TENSOR
    cache = build_layer(f, ctx, table, nb, data.k, data.v, data.k_scale.cpu().numpy(), data.v_scale.cpu().numpy(),
                        gran, bf16_layer)
    window = w.layer_window(layer)
    wid = next(i for i, x in synth.WORKLOADS.items() if x is w)
    if num_splits is None:
        num_splits = WORKLOAD_SPLITS[wid][window]
    out = f.fp8_decode_attn(data.q, cache, to_dev(table), to_dev(ctx), data.q_scale, data.k_scale, data.v_scale,
                            gran, window=window, layer=layer, skip_layer_mask=w.skip_mask(),
                            num_splits=num_splits).float().cpu().numpy()
    cu = np.concatenate([[0], np.cumsum(ctx)])
    qs, ks, vs = (x.cpu().numpy() for x in (data.q_scale, data.k_scale, data.v_scale))
    if num_splits > 0:
        mode = _oracle_mode(w.head_dim, bf16_layer, w.batch, w.num_q_heads, w.num_kv_heads, table.shape[1], window,
                            num_splits)
    else:  # the automatic plan, whose split size the caller derived
        mode = dict(p_quant=True, split_blocks=auto_bps, block_n=decode_block_n(w.head_dim))
    got, ref = [], []
    G = w.group
    for b in seqs:
        T = int(ctx[b])
        for g in sorted(set(h // G for h in heads)):
            hs = [h for h in heads if h // G == g]
            # the whole context at its absolute positions (the window is cut by the oracle)
            kb = synth.bf16_to_f64(data.k[cu[b]:cu[b] + T, g:g + 1])
            vb = synth.bf16_to_f64(data.v[cu[b]:cu[b] + T, g:g + 1])
            qb = synth.bf16_to_f64(data.q[b, g * G:(g + 1) * G])
            sel = lambda a, idx: a if a.size == 1 else a[idx]
            res = attention.decode_attention_contiguous(
                qb, kb, vb, sel(qs, slice(g * G, (g + 1) * G)), sel(ks, slice(g, g + 1)), sel(vs, slice(g, g + 1)),
                fp8=not bf16_layer, window=window, heads=[h - g * G for h in hs], **mode)
            if exact is not None and not bf16_layer:
                pb = attention.decode_attention_contiguous(
                    qb, kb, vb, sel(qs, slice(g * G, (g + 1) * G)), sel(ks, slice(g, g + 1)),
                    sel(vs, slice(g, g + 1)), window=window, heads=[h - g * G for h in hs], p_bound=True)
                exact.extend(pb[h - g * G] for h in hs)
            for h in hs:
                got.append(out[b, h])
                ref.append(res[h - g * G])
    return np.array(got), np.array(ref), data, out


def _exact_check(got, exact, what, record_property):
    o = np.array([e[0] for e in exact])
    bnd = np.array([e[1] for e in exact])
    r, worst = assert_within_p_bound(got, o, bnd, what=what + " vs exact softmax")
    record_property("rel_l2_vs_exact", r)
    record_property("worst_err_over_bound", worst)


def _workload(wid):
    w = synth.WORKLOADS[wid]
    ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
    table, nb = synth.block_table(ctx, seed=w.seed)
    return w, ctx, table, nb


def test_workload_split_counts_give_the_152_sm_plan():
    """The explicit split counts of the workload tests cut the contexts as the automatic
    plan a 152-SM GB300 runs does (the documented rule, restated in the helpers): the
    same blocks per split, or one split either way."""
    for wid, by_window in WORKLOAD_SPLITS.items():
        w, ctx, table, nb = _workload(wid)
        for window, ns in by_window.items():
            n = table.shape[1] if window <= 0 else min(table.shape[1], -(-window // 16) + 1)
            got = decode_split_blocks(table.shape[1], window, ns, w.head_dim)
            want = auto_split_blocks(w.batch, w.num_kv_heads, table.shape[1], window, 152, w.head_dim)
            assert got == want or (got >= n and want >= n), (wid, window, got, want)


def test_workload1_full(record_property):
    w, ctx, table, nb = _workload(1)
    exact = []
    got, ref, _, _ = _decode_layer_check(w, 0, ctx, table, nb, range(w.batch), range(w.num_q_heads), exact=exact)
    assert_close(got, ref, what="workload 1")
    _exact_check(got, exact, "workload 1", record_property)


@pytest.mark.parametrize("layer", [0, 31])
def test_workload2_sampled(layer, record_property):
    w, ctx, table, nb = _workload(2)
    exact = []
    got, ref, _, _ = _decode_layer_check(w, layer, ctx, table, nb, range(w.batch), [0, 5, 13, 22, 31], exact=exact)
    assert_close(got, ref, what=f"workload 2 layer {layer}")
    _exact_check(got, exact, f"workload 2 layer {layer}", record_property)


def test_workload2_automatic_plan_on_152_sms():
    """The benchmark's launch configuration itself (num_splits 0) on a 152-SM GB300: the
    plan must be the hand-derived 208 blocks per split (7 splits), and the output must
    match the oracle walking those splits."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the hand-derived plan is for a 152-SM GB300")
    w, ctx, table, nb = _workload(2)
    assert f.fp8_decode_attn_split_blocks(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, table.shape[1]) == 208
    assert f.fp8_decode_attn_num_splits(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, table.shape[1]) == 7
    got, ref, _, _ = _decode_layer_check(w, 5, ctx, table, nb, range(w.batch), [2, 17, 30], num_splits=0,
                                         auto_bps=208)
    assert_close(got, ref, what="workload 2 automatic plan")


@pytest.mark.parametrize("layer", [0, 1])
def test_workload3_sampled(layer, record_property):
    w, ctx, table, nb = _workload(3)
    exact = []
    got, ref, _, _ = _decode_layer_check(w, layer, ctx, table, nb, range(w.batch), [0, 9, 33, 63], exact=exact)
    assert_close(got, ref, what=f"workload 3 layer {layer}")
    if exact:
        _exact_check(got, exact, f"workload 3 layer {layer}", record_property)


def test_workload4_needle_decode(record_property):
    """128k-key contraction: parity on every head, and each KV group's defining head
    returns the needle's (dequantised) value row."""
    w, ctx, table, nb = _workload(4)
    exact = []
    got, ref, data, out = _decode_layer_check(w, 0, ctx, table, nb, [0], list(range(w.num_q_heads)), exact=exact)
    assert_close(got, ref, what="workload 4 decode")
    _exact_check(got, exact, "workload 4 decode", record_property)
    vs = float(data.v_scale.cpu()[0])
    for g in range(w.num_kv_heads):
        vrow = e4m3.decode(e4m3.quantize(synth.bf16_to_f64(data.v[data.needle_pos, g]), vs)) * vs
        r = np.linalg.norm(out[0, g * w.group] - vrow) / np.linalg.norm(vrow)
        assert r <= 1e-2, f"needle head {g * w.group}: rel_l2 {r:.3e}"


def test_fault_bits_block_id_and_context():
    rng = np.random.default_rng(9)
    ctx = np.array([40, 20], np.int32)
    table, nb = synth.block_table(ctx, seed=1)
    q, k, v = _inputs(rng, ctx, 8, 2, 64)
    one = np.ones(1, np.float32)
    # every pool byte initialised (code 0 = +0.0): the clamped context below reads slots
    # no token was written to, and the output must stay finite
    cache = build_layer(f, ctx, table, nb, k, v, one, one, 0, False, sentinel=0x00)
    bad = table.copy()
    bad[0, 1] = nb + 100
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    f.fp8_decode_attn(q.cuda(), cache, to_dev(bad), to_dev(ctx), to_dev(one), to_dev(one), to_dev(one), 0,
                      fault=fault)
    assert int(fault.item()) & f.FAULT_BLOCK_ID
    fault.zero_()
    long_ctx = np.array([40, 10_000], np.int32)
    o = f.fp8_decode_attn(q.cuda(), cache, to_dev(table), to_dev(long_ctx), to_dev(one), to_dev(one), to_dev(one),
                          0, fault=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) & f.FAULT_CONTEXT
    assert torch.isfinite(o.float()).all()


def test_pipeline_wait_timeout_is_reported_and_the_next_call_is_correct():
    """The timeout path of the tensor-core decode, exercised without a stalled GPU: the
    test hook bounds every pipeline wait at 1 ns, so the first wait not already satisfied
    runs out.  The launch must record FKV_FAULT_TIMEOUT, let its copies and products
    complete (those waits keep their 200 ms bound) and return; its output, merged from a
    zeroed workspace, is finite.  The next call, with the default bound, must reproduce a
    call made before the timeout bit for bit and raise no fault."""
    lib = f.load_library()
    rng = np.random.default_rng(55)
    D, G, Hkv = 128, 4, 2
    Hq = Hkv * G
    ctx = np.array([3000, 700], np.int32)
    table, nb = synth.block_table(ctx, seed=55)
    q, k, v = _inputs(rng, ctx, Hq, Hkv, D)
    one = np.ones(1, np.float32)
    cache = build_layer(f, ctx, table, nb, k, v, one, one, 0, False, sentinel=0xFF)
    ws = f.decode_workspace(len(ctx), Hq, cache, table.shape[1], num_splits=2)
    args = (q.cuda(), cache, to_dev(table), to_dev(ctx), to_dev(one), to_dev(one), to_dev(one), 0)
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = f.fp8_decode_attn(*args, workspace=ws, num_splits=2, fault=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) == 0
    kp, vp = oracle_pools(kvcache, ctx, table, nb, k, v, one, one, False)
    mode = _oracle_mode(D, False, len(ctx), Hq, Hkv, table.shape[1], 0, 2)
    assert_close(ref.float().cpu().numpy(), attention.decode_attention(
        synth.bf16_to_f64(q), kp, vp, table, ctx, one, one, one, **mode), what="before the timeout")
    ws.zero_()
    lib.fkv_set_decode_wait_limit_ns(1)
    try:
        out = f.fp8_decode_attn(*args, workspace=ws, num_splits=2, fault=fault)
        torch.cuda.synchronize()
    finally:
        lib.fkv_set_decode_wait_limit_ns(0)
    assert int(fault.item()) & f.FAULT_TIMEOUT
    assert torch.isfinite(out.float()).all()
    fault.zero_()
    again = f.fp8_decode_attn(*args, workspace=ws, num_splits=2, fault=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) == 0
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))


def test_workspace_counters_are_left_zero_and_checked():
    """The workspace's split counters (its first 4 * batch * num_kv_heads bytes) must be
    zero when a call begins, and every call leaves them zero: consecutive calls on one
    workspace, also with another split plan, give the oracle's results.  A counter that
    is not zero sets FKV_FAULT_WORKSPACE."""
    rng = np.random.default_rng(66)
    D, G, Hkv = 128, 4, 2
    Hq = Hkv * G
    ctx = np.array([2000, 129, 700], np.int32)
    table, nb = synth.block_table(ctx, seed=66)
    q, k, v = _inputs(rng, ctx, Hq, Hkv, D)
    one = np.ones(1, np.float32)
    cache = build_layer(f, ctx, table, nb, k, v, one, one, 0, False, sentinel=0xFF)
    kp, vp = oracle_pools(kvcache, ctx, table, nb, k, v, one, one, False)
    ws = f.decode_workspace(len(ctx), Hq, cache, table.shape[1], num_splits=1)
    ws = torch.zeros(max(ws.numel(), f.fp8_decode_attn_workspace_size(len(ctx), Hq, Hkv, D, table.shape[1], 0, 5)),
                     dtype=torch.uint8, device="cuda")
    counters = ws[:4 * len(ctx) * Hkv].view(torch.int32)
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (q.cuda(), cache, to_dev(table), to_dev(ctx), to_dev(one), to_dev(one), to_dev(one), 0)
    for splits in (5, 2, 5, 1):
        out = f.fp8_decode_attn(*args, workspace=ws, num_splits=splits, fault=fault)
        torch.cuda.synchronize()
        assert int(fault.item()) == 0 and int(counters.abs().sum().item()) == 0
        mode = _oracle_mode(D, False, len(ctx), Hq, Hkv, table.shape[1], 0, splits)
        assert_close(out.float().cpu().numpy(), attention.decode_attention(
            synth.bf16_to_f64(q), kp, vp, table, ctx, one, one, one, **mode), what=f"num_splits={splits}")
    counters[0] = 1000
    f.fp8_decode_attn(*args, workspace=ws, num_splits=2, fault=fault)
    torch.cuda.synchronize()
    assert int(fault.item()) & f.FAULT_WORKSPACE
