// Device helpers shared by the kernels: e4m3 conversions, mbarriers, bulk/TMA copies,
// bounded waits.  sm_103a only.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/fp8kv.h"

#define FKV_DEV __device__ __forceinline__

namespace fkv {

// ---------------------------------------------------------------- fault word

FKV_DEV void raise_fault(int32_t* fault, int32_t bits) {
  if (fault) atomicOr(fault, bits);
}

// ---------------------------------------------------------------- dependent launch

// Programmatic dependent launch: a kernel launched with programmatic stream serialisation
// may start while the kernel before it in the stream is still running.
// griddep_launch_dependents lets the next such kernel's CTAs be scheduled (as this grid's
// CTAs leave the SMs); griddep_wait returns once every earlier grid has completed and its
// memory writes are visible, and precedes every read or write of global memory that an
// earlier kernel may produce or consume.  (Both are no-ops for a plain launch.)
FKV_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
FKV_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- e4m3

// Two float32 values -> two e4m3 codes, round-to-nearest-even, saturating to +-448
// (PTX cvt.rn.satfinite.e4m3x2.f32).  Returns (code(hi) << 8) | code(lo).
FKV_DEV uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two float32 values -> two e5m2 codes, round-to-nearest-even, saturating to +-57344
// (PTX cvt.rn.satfinite.e5m2x2.f32).  Returns (code(hi) << 8) | code(lo).
FKV_DEV uint16_t f32x2_to_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four e5m2 codes (low byte first) -> float32 pairs.  An e5m2 code is the upper byte of
// a binary16, so each code shifted into the high byte of a half is its exact value.
FKV_DEV void e5m2x4_to_f2(uint32_t w, float2& lo, float2& hi) {
  const uint32_t h01 = ((w & 0x000000FFu) << 8) | ((w & 0x0000FF00u) << 16);
  const uint32_t h23 = ((w >> 8) & 0x0000FF00u) | (w & 0xFF000000u);
  lo = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  hi = __half22float2(*reinterpret_cast<const __half2*>(&h23));
}

// Two bf16 packed in a word -> float2 (exact).
FKV_DEV float2 bf16x2_to_f2(uint32_t w) {
  float2 r;
  r.x = __uint_as_float(w << 16);
  r.y = __uint_as_float(w & 0xFFFF0000u);
  return r;
}

// ---------------------------------------------------------------- shared memory / mbarrier

FKV_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

FKV_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

FKV_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

FKV_DEV void mbar_arrive(uint64_t* bar) {
  // the returned state is not needed: the sink operand lets the arrive retire without
  // a result to wait for
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

FKV_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

FKV_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity (never suspends the thread).
FKV_DEV bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same test with a suspend-time hint: a thread whose phase is not complete may sleep up
// to hint_ns before the call returns false.
FKV_DEV bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

FKV_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete, for at most ~timeout_ns of
// wall time.  Returns false on timeout (the caller records a fault and unwinds).
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s

FKV_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, 1000000u)) return true;  // sleep rather than spin
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// One-dimensional bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
FKV_DEV void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

FKV_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier global-memory writes before later async-proxy (TMA) reads.
FKV_DEV void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

FKV_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

FKV_DEV float lg2(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace fkv
