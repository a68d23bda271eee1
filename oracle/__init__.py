"""CPU oracle for FP8 KV-cache quantisation and FP8 attention — TEST INFRASTRUCTURE.

Plain, slow, float64 NumPy restatement of what the hot path computes, written from
the pages (vLLM blog "FP8 KV-Cache and Attention quantization in vLLM" and the
KV-cache explainer "KV Cache量子化とは？").  Only the tests, ``__graft_entry__.smoke``
and the benchmark's CPU-baseline leg may import it; the product library never does,
and it imports nothing from the product library.

Modules and the passages they follow:
  e4m3       the e4m3 codec and scaled quantisation (blog 引言: e4m3 throughout;
             explainer "FP8は値とscaleを組み合わせる": value and scale)
  kvcache    the paged cache write with per-tensor or per-KV-head scales and bf16
             skip layers (blog "Kernel 与 vLLM 改进": Per-Head Scales, 跳过 Layer);
             the KV memory formula (explainer, M_KV = 2 L H_KV D T B S)
  attention  decode attention (unsplit softmax) and prefill attention with the
             kernel's tile walk, P rounded to e4m3 and two-level accumulation
             (blog "Kernel 与 vLLM 改进": Two-level accumulation)

Every function is pinned by tests in ``tests/test_oracle_*.py`` against closed forms,
brute force, invariants or library routines; none is "parity unpinned".
"""
from . import e4m3, kvcache, attention  # noqa: F401
