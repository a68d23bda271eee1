// Blackwell tensor-core helpers (inline PTX, sm_103a): TMEM allocation, tcgen05.mma with
// shared-memory matrix descriptors, commits to mbarriers, TMEM loads/stores, TMA tile loads.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace fkv {

// ---------------------------------------------------------------- TMEM

// Allocate ncols TMEM columns (power of two >= 32); the base address is written to smem.
// Executed by one whole warp.
FKV_DEV void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
FKV_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
FKV_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Per-warpgroup register budgets (setmaxnreg): every warp of the warpgroup executes the same
// instruction.  An increase takes registers that other warpgroups of the CTA have released,
// so the budgets of all warpgroups must add up to no more than the CTA was launched with.
template <int N>
FKV_DEV void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
FKV_DEV void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

FKV_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FKV_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp w reads lanes 32*(w%4)..+31).
FKV_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 lanes from taddr's lane, two halves: threads 0-15 read lanes +0..15 at columns
// [col, col + 32), threads 16-31 the same lanes at columns [col + split, col + split + 32).
template <int SPLIT_COLS>
FKV_DEV void tmem_ld32_16x2(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], %33;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "n"(SPLIT_COLS));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// The store form of tmem_ld32_16x2 with 16 columns: threads 0-15 write lanes +0..15 at
// columns [col, col + 16), threads 16-31 the same lanes at [col + split, col + split + 16).
template <int SPLIT_COLS>
FKV_DEV void tmem_st16_16x2(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %17, {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
               "n"(SPLIT_COLS)
               : "memory");
}
FKV_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive 32-bit TMEM columns of this thread's lane.
FKV_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 consecutive 32-bit TMEM columns of this thread's lane.
FKV_DEV void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

FKV_DEV void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
FKV_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- MMA

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and stride
// byte offsets (all >> 4), version 1, swizzle mode in bits 61..63
// (0 none, 2 128-byte, 4 64-byte, 6 32-byte).
FKV_DEV uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
  return d;
}

// The descriptor of the operand byte_off bytes further on: the start address field holds
// address >> 4 in its low 14 bits, so for shared-memory addresses below 256 KB (every
// offset a multiple of 16) the sum carries into no other field.
FKV_DEV uint64_t desc_add(uint64_t desc, uint32_t byte_off) { return desc + (byte_off >> 4); }

// Instruction descriptor for kind::f8f6f4 with e4m3 A and B, FP32 accumulation.
// a_mn / b_mn: operand stored MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                                    // D format: F32
         | (0u << 7) | (0u << 10)                     // A, B format: E4M3
         | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16)
         | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor for kind::f16 with bf16 A and B, FP32 accumulation.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                                    // D format: F32
         | (1u << 7) | (1u << 10)                     // A, B format: BF16
         | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16)
         | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

FKV_DEV void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
FKV_DEV void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= A B^T with A (M rows = TMEM lanes, K along 32-bit columns, four e4m3 per column)
// read from TMEM at a_tmem and B from shared memory (kind::f8f6f4, FP32 accumulation).
FKV_DEV void umma_f8_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation issued so far by this thread completes.
FKV_DEV void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// One arrival on behalf of the whole (converged) warp: the warp barrier orders every lane's
// earlier writes before lane 0's releasing arrive.  A barrier counted in warps takes 32x
// fewer arrive operations than one counted in threads; each is an update of the same
// shared-memory word, and hundreds of them per tile delay every other barrier operation
// of the CTA (the MMA warp's waits and commits among them).
FKV_DEV void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// ---------------------------------------------------------------- waits

// Pipeline waits of the tensor-core kernels: bounded in wall-clock time (a timeout makes
// the caller record FKV_FAULT_TIMEOUT and drain), sleeping with a suspend-time hint
// rather than spinning.
constexpr uint64_t kPipeWaitNs = 200000000ull;  // 200 ms per wait

// The timed part of a wait.  A bound below the 1 ms suspend hint polls without suspending,
// so that it can run out within its own length.
FKV_DEV bool wait_ns_timed_body(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (limit_ns >= 1000000u ? mbar_try_wait_hint(bar, parity, 1000000u) : mbar_test_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// The same out of line: an inlined wait is then one try_wait and a branch.  In the decode,
// whose MMA and TMA warps pass through many waits per tile, code that a warp runs once per
// tile has to be fetched into the instruction cache again every tile, so their code size
// is their speed.  (A kernel whose warpgroups run under different register budgets takes
// the inline form: one out-of-line function cannot serve callers of different budgets.)
static __device__ __noinline__ bool wait_ns_timed(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return wait_ns_timed_body(bar, parity, limit_ns);
}

// mbarrier.try_wait may itself suspend the thread until the phase completes (for a
// system-dependent time), so a bound below the suspend hint tests without waiting.
template <bool INLINE_SLOW = false>
FKV_DEV bool wait_ns(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kPipeWaitNs) {
  if (limit_ns >= 1000000u ? mbar_try_wait(bar, parity) : mbar_test_wait(bar, parity)) return true;
  if constexpr (INLINE_SLOW) return wait_ns_timed_body(bar, parity, limit_ns);
  else return wait_ns_timed(bar, parity, limit_ns);
}

// Warp-uniform forms: tcgen05.ld / st are warp-collective, so every lane of a warp must
// take the same branch around them.
template <bool INLINE_SLOW = false>
FKV_DEV bool wait_warp(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kPipeWaitNs) {
  const bool ok = wait_ns<INLINE_SLOW>(bar, parity, limit_ns);
  return __all_sync(0xffffffffu, ok);
}
FKV_DEV bool abort_warp(volatile int* flag) { return __any_sync(0xffffffffu, *flag != 0); }


// ---------------------------------------------------------------- TMA

FKV_DEV void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch one tile of a 4-D tensor map into L2 (no shared memory, no completion).
FKV_DEV void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(map), "r"(x), "r"(y),
               "r"(z), "r"(w)
               : "memory");
}

// Host: a 4-D TMA map over one paged pool [num_blocks][Hkv][16][row_bytes] (x = byte in
// the row, slot, KV head, block), uint8 elements, boxes of [16][box_bytes] with the
// 128-byte (box_bytes 128) or 64-byte (box_bytes 64) swizzle.  False when the driver
// entry point is missing or the encoding is rejected.
bool make_pool_map(CUtensorMap* map, void* base, int row_bytes, int Hkv, int num_blocks, int box_bytes);

// Byte offset inside a swizzled tile for a linear (row-major) byte offset: 128-byte swizzle
// XORs address bits 4..6 with bits 7..9, 64-byte swizzle bits 4..5 with bits 7..8 (tile
// bases aligned to 1024 / 512 bytes).
FKV_DEV uint32_t swz(uint32_t lin, int row_bytes) {
  return row_bytes == 128 ? (lin ^ (((lin >> 7) & 7u) << 4)) : (lin ^ (((lin >> 7) & 3u) << 4));
}

}  // namespace fkv
