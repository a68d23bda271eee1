"""fp8_decode_attn_noalloc checked against fp8_decode_attn, through the C ABI.

Callers that cannot hand the library a workspace (a plugin that only receives input and
output pointers from a framework owning all device memory, or a serving loop that must
not call cudaMalloc/cudaFree because those can synchronise the device) use the variant
whose split partials live in the library's fixed device array.  Two calls in a row, with
different shapes so that the second finds the first one's leftovers in the shared
array, must each reproduce the workspace-taking entry point bit for bit: both run the same
kernel with the same split plan, only the scratch's address differs.  One more call goes
through the Python binding of the entry point and must give the same bytes again.

This file is collected last on purpose; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from helpers import build_layer, to_dev

f = pytest.importorskip("fp8_kv_cache_quant_gb300")
pytestmark = pytest.mark.gpu


def _case(D, G, Hkv, ctx, gran, bf16_layer, window, seed):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32)
    table, nb = synth.block_table(ctx, seed=seed)
    n = int(ctx.sum())
    Hq = Hkv * G
    q = torch.from_numpy(rng.standard_normal((len(ctx), Hq, D)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy((rng.standard_normal((n, Hkv, D)) * 2).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    if gran:
        qs, ks, vs = synth.amax_scales(q, 1), synth.amax_scales(k, 1), synth.amax_scales(v, 1)
    else:
        qs = ks = vs = torch.ones(1)
    cache = build_layer(f, ctx, table, nb, k, v, ks.numpy(), vs.numpy(), gran, bf16_layer, sentinel=0xFF)
    return dict(q=q.cuda(), cache=cache, table=to_dev(table), ctx=to_dev(ctx), qs=to_dev(qs), ks=to_dev(ks),
                vs=to_dev(vs), gran=gran, window=window, mask=np.array([1 if bf16_layer else 0], np.uint8))


def _noalloc_c(lib, c, out):
    mask = c["mask"]
    st = lib.fp8_decode_attn_noalloc(
        c["q"].data_ptr(), c["q"].shape[0], c["q"].shape[1], c["cache"].c(), c["table"].data_ptr(),
        c["table"].shape[1], c["ctx"].data_ptr(), c["qs"].data_ptr(), c["ks"].data_ptr(), c["vs"].data_ptr(),
        c["gran"], 0.0, c["window"], 0, mask.ctypes.data, 1, out.data_ptr(), 0, None,
        torch.cuda.current_stream().cuda_stream)
    return st


def test_noalloc_matches_workspace_entry_point_twice():
    lib = f.load_library()
    cases = [
        _case(128, 4, 8, [3000, 45, 700, 16], 1, False, 0, seed=21),
        _case(64, 8, 2, [129, 5000, 1], 0, True, 100, seed=22),
    ]
    for c in cases:
        out = torch.empty_like(c["q"])
        out.fill_(float("nan"))
        assert _noalloc_c(lib, c, out) == f.OK
        ref = f.fp8_decode_attn(c["q"], c["cache"], c["table"], c["ctx"], c["qs"], c["ks"], c["vs"], c["gran"],
                                window=c["window"], skip_layer_mask=c["mask"])
        torch.cuda.synchronize()
        assert torch.isfinite(ref.float()).all()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "noalloc differs from the workspace call"
        # the binding's wrapper of the same entry point (its argument order against the C signature)
        out2 = f.fp8_decode_attn_noalloc(c["q"], c["cache"], c["table"], c["ctx"], c["qs"], c["ks"], c["vs"],
                                         c["gran"], window=c["window"], skip_layer_mask=c["mask"])
        torch.cuda.synchronize()
        assert torch.equal(out2.view(torch.int16), ref.view(torch.int16)), "binding's noalloc differs"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = f.load_library()
    need = f.fp8_decode_attn_workspace_size(512, 32, 8, 128, 8192, 0, 64)
    assert need > f.NOALLOC_WORKSPACE_BYTES
    p = 1 << 12
    cache = f._LayerCache(p, p, 100, 16, 8, 128, 0)
    st = lib.fp8_decode_attn_noalloc(p, 512, 32, cache, p, 8192, p, p, p, p, 0, 0.0, 0, 0, None, 0, p, 64, None,
                                     None)
    assert st == f.INVALID_ARG
