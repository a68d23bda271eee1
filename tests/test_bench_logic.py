"""Host logic of the benchmark (CPU only): ITL fits and break-even against the numbers the
vLLM blog prints (tests/golden/itl_fits.txt), the TTFT quadratic fit and the head_dim-256
ratios (tests/golden/gemma_hd256_fits.txt), byte accounting, the oracle sample of the
reference arm, and the max-over-ranks timing with two gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "itl_fits.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            name, sb, ib, sf, i_f, be, tol, ratio = line.split()
            rows.append((name, float(sb), float(ib), float(sf), float(i_f), float(be), float(tol), float(ratio)))
    return rows


def test_break_even_and_slope_ratio_match_the_blog():
    rows = _golden_rows()
    assert len(rows) == 3
    for name, sb, ib, sf, i_f, be, tol, ratio in rows:
        got = bench.break_even(sf, i_f, sb, ib)
        assert abs(got - be) <= tol * be, (name, got, be)
        assert abs(sf / sb - ratio) <= 0.006, (name, sf / sb, ratio)


def test_gemma_hd256_ratios_match_the_blog():
    """The FP8/BF16 ratios the sweeps report are fp8 over bf16 coefficients, as the blog's."""
    rows = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "gemma_hd256_fits.txt")):
        if line.strip() and not line.startswith("#"):
            name, bf, fp, ratio, tol = line.split()
            rows[name] = (float(bf), float(fp), float(ratio), float(tol))
    for name, (bf, fp, ratio, tol) in rows.items():
        assert abs(fp / bf - ratio) <= tol, (name, fp / bf, ratio)


def test_quadratic_fit_recovers_the_blog_coefficient():
    xs = list(bench.SWEEP_T)
    a, b, c = 1.12e-06, 2.0e-4, 35.0
    ys = [a * x * x + b * x + c for x in xs]
    fa, fb, fc = bench.quadratic_fit(xs, ys)
    assert abs(fa - a) < 1e-12 and abs(fb - b) < 1e-8 and abs(fc - c) < 1e-5
    rng = np.random.default_rng(1)
    noisy = [y * (1 + 1e-3 * e) for y, e in zip(ys, rng.standard_normal(len(xs)))]
    assert abs(bench.quadratic_fit(xs, noisy)[0] / a - 1) < 5e-3


def test_break_even_none_when_fp8_is_not_cheaper():
    assert bench.break_even(2.0, 1.0, 1.0, 0.0) is None


def test_linear_fit_recovers_line():
    xs = [256, 1024, 4096, 16384, 125000]
    ys = [3.2e-3 * x + 41.0 for x in xs]
    s, c = bench.linear_fit(xs, ys)
    assert abs(s - 3.2e-3) < 1e-12 and abs(c - 41.0) < 1e-9
    rng = np.random.default_rng(0)
    ys2 = [y + e for y, e in zip(ys, rng.standard_normal(len(xs)) * 0.01)]
    s2, _ = bench.linear_fit(xs, ys2)
    assert abs(s2 - 3.2e-3) < 1e-6


def test_decode_bytes_accounting():
    w = synth.WORKLOADS[3]
    ctx = np.array([8192, 20000], np.int32)
    import dataclasses
    w2 = dataclasses.replace(w, batch=2)
    per = bench.decode_bytes(w2, ctx, [bool(x) for x in w2.skip_mask()])
    # full layer 0 (e4m3): every key, 2 (K, V) * 8 heads * 64 bytes
    assert per[0]["kv"] == sum(2 * 8 * 64 * int(t) for t in ctx)
    # window layer 1 (bf16, skip mask): the last 128 keys, 2 bytes each
    assert per[1]["kv"] == 2 * (2 * 8 * 64 * 2 * 128)
    assert per[0]["write"] == 2 * 8 * 64 * (2 * 2 + 2 * 1)


def test_oracle_sample_of_the_reference_arm():
    dt, nbytes = bench.oracle_sample(2, 512, 4)
    assert dt > 0 and nbytes == 2 * 1 * 128 * 512


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    bench.dist_barrier(dist, world)
    got = bench.dist_max(dist, world, 1.5 + rank, torch.device("cpu"))
    bench.dist_barrier(dist, world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
    assert res == {0: 2.5, 1: 2.5}


def test_profile_hash_covers_code_not_comments():
    """A committed profile's DRAM figure is trusted while the kernel code is unchanged:
    comments and blank lines do not change the hash, code does."""
    a = "int x = 1;  // one\n/* a block\n   comment */\n\nint y;\n"
    b = "int x = 1;\nint y;   // a reason\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only("int x = 2;") != bench._code_only("int x = 1;")
    assert len(bench.kernel_source_sha("decode_tc.cu")) == 16


def test_profile_hash_covers_the_headers_a_kernel_includes():
    """The hash of a kernel's source takes in the shared headers it includes, directly or
    through another header, and no other: the decode's shared merge code is part of the
    decode kernels' hashes, not of the prefill's or the cache write's."""
    import os
    csrc = os.path.join(bench.ROOT, "fp8_kv_cache_quant_gb300", "csrc")
    tc = bench._local_includes(csrc, "decode_tc.cu")
    assert {"decode_tc.cu", "common.cuh", "tc.cuh", "decode_common.cuh", "kernels.h"} <= tc
    assert "decode_common.cuh" in bench._local_includes(csrc, "decode_attn.cu")
    assert "decode_common.cuh" not in bench._local_includes(csrc, "prefill_attn.cu")
    assert "tc.cuh" not in bench._local_includes(csrc, "kv_quant_cache.cu")
    assert bench.kernel_source_sha("prefill_attn.cu") != bench.kernel_source_sha("decode_tc.cu")


def test_both_arms_describe_the_same_workload_and_sample():
    """The reference arm and the benchmark line's cpu_baseline time the same oracle sample
    and print the same config object."""
    w = synth.WORKLOADS[2]
    keys, heads, text = bench.oracle_sample_shape(2)
    ctx = synth.context_lengths(w.batch, w.ctx_lo, w.ctx_hi, w.seed)
    assert keys == int(ctx[0]) and heads == w.group and str(keys) in text
    a = bench.workload_config(w, ctx, 1)
    b = bench.workload_config(w, ctx, 1, step_bytes=bench._step_bytes_host(w, ctx))
    assert a == b and a["workload"] == w.name and a["context"] == [int(x) for x in ctx]
