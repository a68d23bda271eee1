// Paged GQA decode attention on tcgen05 tensor cores, for e4m3 layers with head_dim 64,
// 128 or 256: split-K over the context, FP8 QK and Score*V products with FP32 accumulation in
// tensor memory, two-level accumulation, FP32 merge of the splits.
//
// The vLLM blog "FP8 KV-Cache and Attention quantization in vLLM": with an FP8 KV cache
// the whole attention runs in FP8, the QK and the Score*V products included (引言); the
// decode is bound by reading the cache ("性能 Benchmark"); each tile's partial result is
// promoted into a true FP32 accumulator ("Kernel 与 vLLM 改进", "Two-level accumulation").
//
// A decode step has one query per sequence, so a (sequence, KV head) contributes only G
// query rows.  The products are therefore taken transposed, with the keys and head_dim on
// the MMA's M side and the G query heads (padded to 16) on N:
//   S^T [128 keys][16]   = K8 [128 keys][D]   . Q8^T [D][16]        (K, Q8 K-major)
//   O^T [128 d][16]     += V8^T [128 d][BN keys] . P8^T [BN keys][16]   (V MN-major)
// so the cache tiles are the A operands exactly as TMA lands them from the pool.
// head_dim 64 uses 64-byte rows (64-byte swizzle), tiles of BN = 256 keys (two S^T
// products of 128 keys; a tile's fixed costs, the softmax's reductions and barriers and
// the products' latencies, then serve twice the bytes), and an M = 64 P.V product, whose
// accumulator row r sits in TMEM lane 32 (r / 16) + r % 16.  Other head_dims: BN = 128.
//
// CTA = (split, KV head g, sequence b), 10 warps:
//   warps 0-3  softmax: quantise the G query rows to e4m3 (prologue); per tile thread i
//              owns key i (and 128 + i at head_dim 64; TMEM lane i): S^T row from TMEM, scale, mask,
//              per-head tile maximum across the 128 keys (shuffles + shared memory),
//              running max m, p = 2^(s - m), its unrounded sum, P8 = e4m3(p * 448) into
//              the P^T tile; the tile's alpha = 2^(m_old - m) is published in shared memory.
//   warps 4-7  correction: thread i owns head_dim row i (and 128 + i): each tile's
//              O_tile^T is promoted into FP32 registers, acc = acc * alpha + O_tile, off
//              the softmax warps' critical path; then the split's output.
//   warp 8     K copies: each 16-token block is one box [16][row bytes] of the paged pool
//              (4-D tensor map), a tile's BN / 16 blocks issued from as many lanes; in the prologue
//              also the first tiles' V copies, and (fp8_decode_step) the current token's
//              K and V written into the pools by the split that holds it.
//   warp 9     allocates TMEM; polls the pipeline's barriers and issues whichever is ready
//              of a V tile's copies (8 lanes), an S^T product (one tile ahead) and a P.V
//              product, committing to mbarriers.
// The split writes (o / l, log2-sum-exp) per head; the CTA that finishes the last split
// of (b, g) merges all of them in FP32.  Every wait is bounded in time (the pipeline's by
// p.pipe_wait_ns); a timeout records FKV_FAULT_TIMEOUT, lets the CTA's copies and MMAs
// drain (those waits keep the fixed bound kPipeWaitNs) and returns.
#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace fkv {
namespace {

template <int D, int G>
struct DecodeTcCfg {
  static constexpr int BN = D == 64 ? 256 : 128;  // keys per tile (the P rounding's tile)
  static constexpr int TPB = BN / 16;             // pool blocks per tile
  static constexpr int NHALF = BN / 128;          // S^T products (M = 128 keys each) per tile
  static constexpr int NP = 16;                // query heads padded to the MMA's N
  static constexpr int RB = D < 128 ? D : 128; // bytes of one swizzled row
  static constexpr int SWZ = RB == 128 ? 2 : 4;  // descriptor swizzle mode (128 / 64 bytes)
  static constexpr int NSUB = D / RB;          // column blocks of a K / V row
  static constexpr int KSUB = BN * RB;         // bytes of one column block of a K / V tile
  static constexpr int KTILE = BN * D;         // bytes of a K or V tile
  static constexpr int MPV = D < 128 ? D : 128;  // M of one P.V product (head_dim rows)
  static constexpr int NS = 2;                 // K / V stages (small CTAs: 3 per SM up to head_dim 128)
  static constexpr int MAX_BPS = kMaxSplitBlocks;          // blocks per split
  static constexpr int QSUB = NP * RB;         // bytes of one column block of the Q8 tile
  static constexpr int PTILE = NP * BN;        // bytes of one P8^T tile: NHALF sub-tiles [NP][128 keys]
  static constexpr int TM_S = 0;               // S^T buffers: TMEM columns [0, 2 * NHALF * NP)
  static constexpr int TM_O = 2 * NHALF * NP;  // O_tile^T buffers: [TM_O, TM_O + 2 * NSUB * NP)
  static constexpr int SLD = (D == 64 && G <= 8) ? 8 : 16;  // S^T columns a softmax thread loads
  // block ids of the split staged in shared memory once (head_dim 128 and 256); at head_dim
  // 64, whose three CTAs per SM leave no room for them, each copying lane reads its block's
  // id one tile ahead of the copy
  static constexpr bool STAGE_IDS = D != 64;
  static constexpr int TM_COLS = TM_O + 2 * NSUB * NP <= 64 ? 64 : 128;
  // shared memory (bytes; tiles on 1024-byte boundaries for the 128-byte swizzle)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NS * KTILE;
  static constexpr int OFF_Q = OFF_V + NS * KTILE;
  static constexpr int OFF_P = OFF_Q + NSUB * QSUB;  // two P8^T tiles
  static constexpr int OFF_RED = OFF_P + 2 * PTILE;  // [2][4 warps][NP] floats
  static constexpr int OFF_A = OFF_RED + 2 * 4 * NP * 4;  // alpha [2][NP]; then m, l [2][NP]
  static constexpr int OFF_BAR = OFF_A + 4 * NP * 4;
  static constexpr int NBAR = 21 + 4 * NS;
  static constexpr int OFF_IDS = OFF_BAR + NBAR * 8;     // [MAX_BPS] block ids of the split (STAGE_IDS)
  static constexpr int OFF_MISC = OFF_IDS + (STAGE_IDS ? MAX_BPS * 4 : 0);
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t IDESC_QK = idesc_e4m3_f32(128, NP, 0, 0);  // K8 and Q8 K-major
  static constexpr uint32_t IDESC_PV = idesc_e4m3_f32(MPV, NP, 1, 0);  // V8 MN-major, P8 K-major
  // merge scratch (in the K stages, free by then): 2 G + G * CH floats
  static constexpr int CH = (NS * KTILE / 4 - 2 * G) / G < 256 ? (NS * KTILE / 4 - 2 * G) / G : 256;
  static_assert(G >= 1 && G <= NP, "query heads per KV head");
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
  static_assert(MAX_BPS % TPB == 0 && TPB * NS <= 32, "whole tiles per split; the prologue's ids in one warp");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // three CTAs per SM up to head_dim 128 (G <= 8): each takes SMEM plus 1 KB the hardware
  // reserves, out of the SM's 228 KB
  static_assert(D > 128 || G > 8 || 3 * (SMEM + 1024) <= 228 * 1024, "three CTAs per SM");
};

constexpr int kDecodeTcThreads = 320;  // softmax warpgroup, correction warpgroup, TMA warp, MMA warp

// The current token's K and V row of KV head g, written into the e4m3 pools at position
// T - 1 exactly as kv_quant_cache writes them: e4m3(fl32(x * fl32(1 / s))), round to
// nearest even, saturating.  One warp; lane j < 2 D / 8 takes 8 elements of K (j < D / 8)
// or V.  The fence orders the writes before the TMA copies that read the block back.
template <int D>
__device__ void write_current_token(const DecodeParams& p, int b, int g, int T, int lane) {
  const int pos = T - 1;
  const int id = p.block_table[static_cast<size_t>(b) * p.max_blocks + (pos >> 4)];
  if (id < 0 || id >= p.num_blocks) return;  // reported by the block-id checks of the split
  const size_t row = ((static_cast<size_t>(id) * p.Hkv + g) * 16 + (pos & 15)) * D;  // byte offset
  const size_t src = (static_cast<size_t>(b) * p.Hkv + g) * D;
  constexpr int CH = D / 8;
  for (int j = lane; j < 2 * CH; j += 32) {
    const bool is_v = j >= CH;
    const int c = is_v ? j - CH : j;
    const uint4 x = reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) + src)[c];
    const float inv = __frcp_rn((is_v ? p.v_scale : p.k_scale)[p.per_head ? g : 0]);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 f0 = bf16x2_to_f2(w[2 * k]), f1 = bf16x2_to_f2(w[2 * k + 1]);
      o[k] = static_cast<uint32_t>(f32x2_to_e4m3x2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv))) |
             (static_cast<uint32_t>(f32x2_to_e4m3x2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv))) << 16);
    }
    // the pools are the caller's writable device memory; the params carry them as const
    // because the plain decode only reads them
    uint8_t* dst = const_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) + row + 8 * c;
    *reinterpret_cast<uint2*>(dst) = make_uint2(o[0], o[1]);
  }
  fence_proxy_async_global();
}

// Maximum of a value over the 32 lanes of a warp, in one warp-wide reduction (every lane
// takes part and receives the result).
FKV_DEV float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

template <int D, int G>
__global__ void __launch_bounds__(kDecodeTcThreads, (D <= 128 && G <= 8) ? 3 : 1)
    decode_tc_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  using C = DecodeTcCfg<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sP = smem + C::OFF_P;
  float* red_s = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_A);  // [2][NP] alpha of tile t in slot t % 2
  float* ml_s = alpha_s + 2 * C::NP;                           // [2][NP] the split's m and l
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;    // [2] S^T(t) in buffer t % 2
  uint64_t* s_free = bars + 3;    // [2]
  uint64_t* p_full = bars + 5;    // [2] P8^T(t) in tile t % 2
  uint64_t* p_free = bars + 7;    // [2]
  uint64_t* o_full = bars + 9;    // [2] O_tile^T(t) in buffer t % 2
  uint64_t* o_free = bars + 11;   // [2]
  uint64_t* mma_done = bars + 13;
  uint64_t* red_full = bars + 14;  // [2] the 4 warps' per-head values of reduction r in slot r % 2
  uint64_t* a_full = bars + 16;    // [2] alpha of tile t published in slot t % 2
  uint64_t* a_free = bars + 18;    // [2] ... and read by the correction warpgroup
  uint64_t* l_full = bars + 20;    // the split's m and l published
  uint64_t* k_full = bars + 21;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* v_full = k_empty + C::NS;
  uint64_t* v_empty = v_full + C::NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* last_s = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  int* ids_s = reinterpret_cast<int*>(smem + C::OFF_IDS);

  const int sigma = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The next kernel in the stream may be scheduled as this grid's CTAs finish.  The
  // barriers and the tensor memory need no input, so they are set up before waiting for
  // the kernels before this one (their writes to the inputs, the pools and the workspace).
  griddep_launch_dependents();
  if (warp == 8 && lane == 0) {
    // barriers signalled by the softmax or correction warps count warps (one arrival each)
    mbar_init(q_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_free[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 4);
    }
    mbar_init(mma_done, 1);
    mbar_init(&red_full[0], 4);
    mbar_init(&red_full[1], 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&a_free[i], 4);
    }
    mbar_init(l_full, 4);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    *abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  constexpr int TPB = C::TPB;
  griddep_wait();
  // Without a window a split's blocks start at sigma * bps whatever the context length,
  // so the producer warp reads its first tiles' table entries alongside the length
  // (entries past the sequence's blocks are read but not used).
  int id_spec = 0;
  if (warp == 8 && p.window <= 0 && lane < TPB * C::NS && sigma * p.bps + lane < p.max_blocks)
    id_spec = p.block_table[static_cast<size_t>(b) * p.max_blocks + sigma * p.bps + lane];
  const SeqRange r = seq_range(p, b, sigma == 0 && g == 0 && threadIdx.x == 0);
  if (sigma >= r.nsplit) {  // uniform over the CTA
    if (sigma == 0) {       // a sequence without keys: zero output rows
      for (int t = threadIdx.x; t < G * D; t += blockDim.x)
        p.out[(static_cast<size_t>(b) * p.Hq + g * G + t / D) * D + t % D] = __float2bfloat16(0.f);
    }
    __syncthreads();
    if (warp == 9) {
      tc_fence_after();
      tmem_dealloc(*tmem_slot, C::TM_COLS);
    }
    return;
  }
  // this split: blocks [bb, be), keys [klo, khi), tiles of TPB blocks from block bb
  const int bb = r.blk_begin + sigma * p.bps;
  const int be = min(bb + p.bps, r.blk_end);
  const int klo = max(r.lo, bb * 16), khi = min(r.T, be * 16);
  const int n_t = (be - bb + TPB - 1) / TPB;
  const int T = r.T;
  // block id of block j of the split (an id out of range reads block 0 and is reported)
  auto checked_block_id = [&](int id) -> int {
    if (id < 0 || id >= p.num_blocks) {
      raise_fault(p.fault, FKV_FAULT_BLOCK_ID);
      id = 0;
    }
    return id;
  };
  auto split_block_id = [&](int j) -> int {
    if (j >= be - bb) return 0;
    return checked_block_id(p.block_table[static_cast<size_t>(b) * p.max_blocks + bb + j]);
  };

  // Before the CTA-wide barrier the K-producer warp issues the K and V copies of the first
  // NS tiles, so that the first HBM latency overlaps the rest of the prologue (block-id
  // staging, the query's quantisation).
  const int n0 = min(C::NS, n_t);  // tiles whose copies go out in the prologue
  // fp8_decode_step: the split holding position T - 1 (the last) writes the current token
  // into the pools before its first copy of that block (not when the context was clamped)
  if (warp == 8 && p.k_new != nullptr && sigma == r.nsplit - 1 && !r.clamped) write_current_token<D>(p, b, g, T, lane);
  if (warp == 8) {
    __syncwarp();
    int id = 0;  // block `lane` of the split
    if (lane < TPB * n0)
      id = p.window > 0 ? split_block_id(lane) : (lane < be - bb ? checked_block_id(id_spec) : 0);
    if (C::STAGE_IDS && lane < TPB * n0) ids_s[lane] = id;
    for (int t = 0; t < n0; ++t) {
      const int nblk = min(TPB, be - bb - TPB * t);
      const int idt = __shfl_sync(0xffffffffu, id, TPB * t + (lane & (TPB - 1)));
      if (lane == 0) {
        mbar_arrive_expect_tx(&k_full[t], nblk * 16 * D);
        mbar_arrive_expect_tx(&v_full[t], nblk * 16 * D);
      }
      __syncwarp();
      if (lane < nblk) {
#pragma unroll
        for (int s = 0; s < C::NSUB; ++s) {
          tma_load_4d(sK + t * C::KTILE + s * C::KSUB + lane * 16 * C::RB, &tmk, s * C::RB, 0, g, idt, &k_full[t]);
          tma_load_4d(sV + t * C::KTILE + s * C::KSUB + lane * 16 * C::RB, &tmv, s * C::RB, 0, g, idt, &v_full[t]);
        }
      }
    }
  }
  if constexpr (C::STAGE_IDS) {
    // the split's other block ids, checked once
    for (int j = TPB * n0 + threadIdx.x; j < be - bb; j += blockDim.x) ids_s[j] = split_block_id(j);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ============================================================ softmax warpgroup
    const int i = threadIdx.x;  // key i of a tile (TMEM lane i)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // ---- prologue: the G query rows -> e4m3 codes in the swizzled Q8 tile (rows G..15
    // zero), and the padding rows of both P8^T tiles zeroed once
    {
      const int row = i >> 3;
#pragma unroll
      for (int c = i & 7; c < D / 16; c += 8) {
        uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
        if (row < G) {
          const int h = g * G + row;
          const float iq = __frcp_rn(p.q_scale[p.per_head ? h : 0]);
          const uint4* src = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.Hq + h) * D) + 2 * c;
          const uint4 a = src[0], a2 = src[1];
          const uint32_t in[8] = {a.x, a.y, a.z, a.w, a2.x, a2.y, a2.z, a2.w};
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 x0 = bf16x2_to_f2(in[2 * j]), x1 = bf16x2_to_f2(in[2 * j + 1]);
            w[j] = static_cast<uint32_t>(f32x2_to_e4m3x2(__fmul_rn(x0.x, iq), __fmul_rn(x0.y, iq))) |
                   (static_cast<uint32_t>(f32x2_to_e4m3x2(__fmul_rn(x1.x, iq), __fmul_rn(x1.y, iq))) << 16);
          }
          w4 = make_uint4(w[0], w[1], w[2], w[3]);
        }
        const int byte = c * 16;
        *reinterpret_cast<uint4*>(sQ + (byte / C::RB) * C::QSUB +
                                  swz(static_cast<uint32_t>(row * C::RB + byte % C::RB), C::RB)) = w4;
      }
      if constexpr (G < C::NP) {
        constexpr int PAD = (C::NP - G) * 8;  // 16-byte chunks of one sub-tile's padding rows
        for (int x = i; x < 2 * C::NHALF * PAD; x += 128) {
          const int sub = x / PAD, rem = x % PAD;  // sub-tile (tile * NHALF + half)
          *reinterpret_cast<uint4*>(sP + (sub / C::NHALF) * C::PTILE + (sub % C::NHALF) * (C::NP * 128) +
                                    (G + rem / 8) * 128 + (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(q_full);
    }
    float cst[G];  // log2(e) * softmax scale * q_s[h] * k_s[g]
#pragma unroll
    for (int h = 0; h < G; ++h)
      cst[h] = p.sm_scale_log2 * p.q_scale[p.per_head ? g * G + h : 0] * p.k_scale[p.per_head ? g : 0];
    float m[G], lsum[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      lsum[h] = 0.f;
    }
    bool ok = true;
    for (int t = 0; t < n_t; ++t) {
      if ((t & 7) == 7 && abort_warp(abort_s)) { ok = false; break; }
      const int sb = t & 1;
      if (!wait_warp(&s_full[sb], (t >> 1) & 1, p.pipe_wait_ns)) { ok = false; break; }
      tc_fence_after();
      constexpr int NH2 = C::NHALF;
      float sv[NH2][C::SLD];  // key i + 128 hh of the tile: S^T product hh, lane i
#pragma unroll
      for (int hh = 0; hh < NH2; ++hh) {
        const uint32_t col = lane_base + C::TM_S + (sb * NH2 + hh) * C::NP;
        if constexpr (C::SLD == 8) tmem_ld8(col, sv[hh]);
        else tmem_ld16(col, sv[hh]);
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive_warp(&s_free[sb]);
      bool valid[NH2];
      float x[NH2][G], wm[G];
#pragma unroll
      for (int hh = 0; hh < NH2; ++hh) {
        const int key = (bb + TPB * t) * 16 + 128 * hh + i;
        valid[hh] = key >= klo && key < khi;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int hh = 0; hh < NH2; ++hh) x[hh][h] = valid[hh] ? sv[hh][h] * cst[h] : -INFINITY;
        wm[h] = x[0][h];
#pragma unroll
        for (int hh = 1; hh < NH2; ++hh) wm[h] = fmaxf(wm[h], x[hh][h]);
      }
      // tile maximum of each head over the tile's keys: within the warp (one warp-wide
      // reduction per head), then across the 4
#pragma unroll
      for (int h = 0; h < G; ++h) wm[h] = warp_max(wm[h]);
      // reduction t uses slot t % 2 (its previous use, t - 2, was read by every warp
      // before that warp's arrival for t - 1)
      float* red = red_s + (t & 1) * 4 * C::NP;
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) red[warp * C::NP + h] = wm[h];
        mbar_arrive(&red_full[t & 1]);
      }
      if (!wait_warp(&red_full[t & 1], (t >> 1) & 1, p.pipe_wait_ns)) { ok = false; break; }
      const int pb = t & 1;
      // P8^T tile t % 2 is free once the P.V of tile t-2 completed; alpha slot t % 2 once
      // the correction warpgroup read tile t-2's alpha
      if (t >= 2 && !wait_warp(&p_free[pb], ((t >> 1) - 1) & 1, p.pipe_wait_ns)) { ok = false; break; }
      if (t >= 2 && !wait_warp(&a_free[pb], ((t >> 1) - 1) & 1, p.pipe_wait_ns)) { ok = false; break; }
      float pvs[NH2][G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float tmax = fmaxf(fmaxf(red[h], red[C::NP + h]), fmaxf(red[2 * C::NP + h], red[3 * C::NP + h]));
        const float mn = fmaxf(m[h], tmax);
        const float alpha = (m[h] == -INFINITY) ? 0.f : ex2(m[h] - mn);
        float psum = 0.f;
#pragma unroll
        for (int hh = 0; hh < NH2; ++hh) {
          const float pv = valid[hh] ? ex2(x[hh][h] - mn) : 0.f;
          psum = hh == 0 ? pv : psum + pv;
          pvs[hh][h] = pv * 448.f;
        }
        lsum[h] = fmaf(lsum[h], alpha, psum);
        m[h] = mn;
        if (i == 0) alpha_s[pb * C::NP + h] = alpha;
      }
      // P8 codes, two heads per conversion
#pragma unroll
      for (int hh = 0; hh < NH2; ++hh) {
#pragma unroll
        for (int h = 0; h < G; h += 2) {
          const uint16_t code2 = f32x2_to_e4m3x2(pvs[hh][h], h + 1 < G ? pvs[hh][h + 1] : 0.f);
          uint8_t* row = sP + pb * C::PTILE + hh * (C::NP * 128);
          row[swz(static_cast<uint32_t>(h * 128 + i), 128)] = static_cast<uint8_t>(code2 & 0xFF);
          if (h + 1 < G) row[swz(static_cast<uint32_t>((h + 1) * 128 + i), 128)] = static_cast<uint8_t>(code2 >> 8);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(&p_full[pb]);
      mbar_arrive_warp(&a_full[pb]);
    }
    if (!ok) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      *abort_s = 1;
    }
    // ---- the split's l (summed over the 128 key threads: reduction n_t) and m, published
    // for the correction warpgroup
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int h = 0; h < G; ++h) lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], off);
    float* red = red_s + (n_t & 1) * 4 * C::NP;
    if (ok && lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) red[warp * C::NP + h] = lsum[h];
      mbar_arrive(&red_full[n_t & 1]);
    }
    if (ok && !wait_warp(&red_full[n_t & 1], (n_t >> 1) & 1, p.pipe_wait_ns)) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      *abort_s = 1;
      ok = false;
    }
    if (ok && i == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        ml_s[h] = m[h];
        ml_s[C::NP + h] = (red[h] + red[C::NP + h]) + (red[2 * C::NP + h] + red[3 * C::NP + h]);
      }
    }
    if (ok) mbar_arrive_warp(l_full);
  } else if (warp < 8) {
    // ============================================================ correction warpgroup
    const int i = threadIdx.x - 128;  // TMEM lane i
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp - 4) * 32) << 16);
    // the head_dim row this lane holds (and 128 + it): lane i itself for M = 128; for the
    // M = 64 product of head_dim 64, lanes 0-15 of each warp hold rows 16 (warp - 4) + lane
    const bool has_row = C::MPV == 128 || lane < 16;
    const int d = C::MPV == 128 ? i : (warp - 4) * 16 + lane;
    float acc[C::NSUB][G];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int s2 = 0; s2 < C::NSUB; ++s2) acc[s2][h] = 0.f;
    bool ok = true;
    for (int t = 0; t < n_t; ++t) {
      if ((t & 7) == 7 && abort_warp(abort_s)) { ok = false; break; }
      const int ob = t & 1;
      if (!wait_warp(&a_full[ob], (t >> 1) & 1, p.pipe_wait_ns)) { ok = false; break; }
      float alpha[G];
#pragma unroll
      for (int h = 0; h < G; ++h) alpha[h] = alpha_s[ob * C::NP + h];
      mbar_arrive_warp(&a_free[ob]);
      // acc = acc * alpha + O_tile^T(t): the two-level accumulation of tile t
      if (!wait_warp(&o_full[ob], (t >> 1) & 1, p.pipe_wait_ns)) { ok = false; break; }
      tc_fence_after();
      float o[C::NSUB][16];
#pragma unroll
      for (int s2 = 0; s2 < C::NSUB; ++s2) tmem_ld16(lane_base + C::TM_O + (ob * C::NSUB + s2) * C::NP, o[s2]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive_warp(&o_free[ob]);
#pragma unroll
      for (int s2 = 0; s2 < C::NSUB; ++s2)
#pragma unroll
        for (int h = 0; h < G; ++h) acc[s2][h] = fmaf(acc[s2][h], alpha[h], o[s2][h]);
    }
    if (!ok) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      *abort_s = 1;
    }
    // ---- this split's result: o = acc / (448 l) and lse = m + log2(l) per head
    if (ok && wait_warp(l_full, 0, p.pipe_wait_ns)) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float L = ml_s[C::NP + h];
        const size_t row = (static_cast<size_t>(b) * p.Hq + g * G + h) * p.max_splits + sigma;
        const float inv = L > 0.f ? 1.f / (448.f * L) : 0.f;  // P8 carries the factor 448
        if (has_row) {
#pragma unroll
          for (int s2 = 0; s2 < C::NSUB; ++s2) p.o_part[row * D + s2 * 128 + d] = acc[s2][h] * inv;
        }
        if (i == 0) p.lse_part[row] = L > 0.f ? ml_s[h] + lg2(L) : -INFINITY;
      }
    } else if (ok) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
    }
  } else if (warp == 8) {
    // ============================================================ TMA producer of K
    // K(t) into stage t % NS once the S^T of tile t - NS has read it; blocks past the
    // split are not loaded (their keys are masked)
    // Lane j issues block j's copies: copies issued from one thread serialise (a
    // thread waiting on one copy issues no other), so the tile's 8 blocks go out from 8
    // lanes at once.
    int last_use[C::NS];
#pragma unroll
    for (int s = 0; s < C::NS; ++s) last_use[s] = s < n0 ? 0 : -1;  // the prologue's copies
    // (head_dim 64: block `lane` of tile n0, read ahead)
    int kid = (!C::STAGE_IDS && lane < TPB) ? split_block_id(TPB * n0 + lane) : 0;
    for (int t = n0; t < n_t; ++t) {
      if (abort_warp(abort_s)) break;
      const int st = t % C::NS, use = t / C::NS;
      if (use > 0 && !wait_warp(&k_empty[st], (use - 1) & 1, p.pipe_wait_ns)) {
        if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
        *abort_s = 1;
        break;
      }
      const int nblk = min(TPB, be - bb - TPB * t);
      int id_t = kid;
      if constexpr (C::STAGE_IDS) {
        id_t = lane < TPB ? ids_s[TPB * t + lane] : 0;
      } else {
        kid = lane < TPB ? split_block_id(TPB * (t + 1) + lane) : 0;  // the next tile's, read meanwhile
      }
      if (lane == 0) mbar_arrive_expect_tx(&k_full[st], nblk * 16 * D);
      __syncwarp();
      if (lane < nblk) {
#pragma unroll
        for (int s = 0; s < C::NSUB; ++s)
          tma_load_4d(sK + st * C::KTILE + s * C::KSUB + lane * 16 * C::RB, &tmk, s * C::RB, 0, g, id_t, &k_full[st]);
      }
      last_use[st] = use;
    }
    // let every issued copy land before the CTA can exit
    if (lane == 0)
      for (int s = 0; s < C::NS; ++s)
        if (last_use[s] >= 0) wait_ns(&k_full[s], last_use[s] & 1);
    __syncwarp();
  } else {
    // ============================================================ MMA issuer and V producer (warp 9)
    // Lane 0 polls the pipeline's barriers without blocking and issues, in whatever order
    // they become possible, the V loads, the S^T products and the P.V products, so that
    // a late K tile never holds back a P.V (and the V stage it frees) or vice versa.
    const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV), sPa = smem_u32(sP);
    int tq = 0, tp = 0, tv = n0;  // next S^T, P.V and V load to issue (the first n0 V loads: prologue)
    int v_last[C::NS];
#pragma unroll
    for (int s = 0; s < C::NS; ++s) v_last[s] = s < n0 ? 0 : -1;
    // (head_dim 64: block `lane` of tile tv, read ahead)
    int vid = (!C::STAGE_IDS && lane < TPB) ? split_block_id(TPB * tv + lane) : 0;
    bool ok = wait_warp(q_full, 0, p.pipe_wait_ns);
    uint64_t t_progress = globaltimer_ns();
    while (ok && tp < n_t) {
      if (abort_warp(abort_s)) break;
      int events = 0;  // bit 0: progress; bit 1: P.V of tile tp ready; bit 2: V(tv) may load
      // V(tv) into stage tv % NS once the P.V of tile tv - NS has read it (lane j issues
      // block j's copy)
      int vgo = 0;
      if (lane == 0)
        vgo = tv < n_t && (tv < C::NS || mbar_test_wait(&v_empty[tv % C::NS], ((tv / C::NS) - 1) & 1));
      if (__shfl_sync(0xffffffffu, vgo, 0)) {
        const int st = tv % C::NS;
        const int nblk = min(TPB, be - bb - TPB * tv);
        if (lane == 0) mbar_arrive_expect_tx(&v_full[st], nblk * 16 * D);
        __syncwarp();
        if constexpr (C::STAGE_IDS) vid = lane < TPB ? ids_s[TPB * tv + lane] : 0;
        if (lane < nblk) {
#pragma unroll
          for (int s = 0; s < C::NSUB; ++s)
            tma_load_4d(sV + st * C::KTILE + s * C::KSUB + lane * 16 * C::RB, &tmv, s * C::RB, 0, g, vid, &v_full[st]);
        }
        v_last[st] = tv / C::NS;
        ++tv;
        if constexpr (!C::STAGE_IDS) vid = lane < TPB ? split_block_id(TPB * tv + lane) : 0;  // the next tile's
        events |= 1;
      }
      if (lane == 0) {
        // S^T(tq) = K8(tq) Q8^T into S buffer tq % 2: K landed, the buffer's previous S read
        if (tq < n_t && mbar_test_wait(&k_full[tq % C::NS], (tq / C::NS) & 1) &&
            (tq < 2 || mbar_test_wait(&s_free[tq & 1], ((tq >> 1) - 1) & 1))) {
          const int st = tq % C::NS, sb = tq & 1;
          tc_fence_after();
          // one product per 128 keys of the tile (rows 128 hh .. of the K tile)
#pragma unroll
          for (int hh = 0; hh < C::NHALF; ++hh)
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              const int byte = kk * 32;
              const uint64_t ad = smem_desc(sKa + st * C::KTILE + (byte / C::RB) * C::KSUB + hh * 128 * C::RB +
                                                byte % C::RB,
                                            16, 8 * C::RB, C::SWZ);
              const uint64_t bd = smem_desc(sQa + (byte / C::RB) * C::QSUB + byte % C::RB, 16, 8 * C::RB, C::SWZ);
              umma_f8(tmem + C::TM_S + (sb * C::NHALF + hh) * C::NP, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
            }
          umma_commit(&s_full[sb]);
          umma_commit(&k_empty[st]);
          ++tq;
          events |= 1;
        }
        // P.V of tile tp: P written, V landed, the O_tile buffer promoted (tile tp - 2)
        if (tp < tq && mbar_test_wait(&p_full[tp & 1], (tp >> 1) & 1) &&
            mbar_test_wait(&v_full[tp % C::NS], (tp / C::NS) & 1) &&
            (tp < 2 || mbar_test_wait(&o_free[tp & 1], ((tp >> 1) - 1) & 1)))
          events |= 2;
      }
      events = __shfl_sync(0xffffffffu, events, 0);
      if (events & 2) {
        const int st = tp % C::NS, pb = tp & 1;
        // keys past the context may hold stale bytes (NaN codes) or were not loaded: zero
        // their V rows, since 0 * NaN would poison the product even though their P is 0
        const int kbase = (bb + TPB * tp) * 16;
        if (kbase + C::BN > T) {
          const int first = max(T - kbase, 0);
          constexpr int CPR = C::RB / 16;  // 16-byte chunks per row
          const int items = (C::BN - first) * C::NSUB * CPR;
          for (int it = lane; it < items; it += 32) {
            const int c = it % CPR;
            const int s = (it / CPR) % C::NSUB;
            const int rr = first + (it / CPR) / C::NSUB;
            *reinterpret_cast<uint4*>(sV + st * C::KTILE + s * C::KSUB + rr * C::RB + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          // O_tile^T(tp) = V8(tp)^T P8(tp)^T into O buffer tp % 2, one M = 128 product per column block
#pragma unroll
          for (int s = 0; s < C::NSUB; ++s)
#pragma unroll
            for (int kk = 0; kk < C::BN / 32; ++kk) {
              const uint64_t ad = smem_desc(sVa + st * C::KTILE + s * C::KSUB + kk * 32 * C::RB, 8 * C::RB, 8 * C::RB,
                                            C::SWZ);
              // keys 32 kk ..: sub-tile kk / 4 of P8^T, 32 bytes into its 128-byte rows
              const uint64_t bd = smem_desc(sPa + pb * C::PTILE + (kk / 4) * (C::NP * 128) + (kk % 4) * 32, 16, 1024, 2);
              umma_f8(tmem + C::TM_O + (pb * C::NSUB + s) * C::NP, ad, bd, C::IDESC_PV, kk > 0 ? 1u : 0u);
            }
          umma_commit(&o_full[pb]);
          umma_commit(&v_empty[st]);
          umma_commit(&p_free[pb]);
        }
        __syncwarp();
        ++tp;
      }
      if (events != 0) {
        t_progress = globaltimer_ns();
      } else if (globaltimer_ns() - t_progress > p.pipe_wait_ns) {
        ok = false;
      } else {
        __nanosleep(32);  // leave the issue slots to the softmax warp sharing this SM quarter
      }
    }
    if (!ok) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      *abort_s = 1;
    }
    // every MMA issued by this warp completes before TMEM is released, and every V copy
    // lands before the CTA can exit
    if (lane == 0) {
      umma_commit(mma_done);
      wait_ns(mma_done, 0);
      for (int s = 0; s < C::NS; ++s)
        if (v_last[s] >= 0) wait_ns(&v_full[s], v_last[s] & 1);
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }

  // ---------------------------------------------------- the last split of (b, g) merges
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *last_s = count_split_done(p, b * p.Hkv + g, r.nsplit);
  __syncthreads();
  if (!*last_s) return;
  __threadfence();
  merge_splits<D, G, kDecodeTcThreads, C::CH>(p, b, g, r.nsplit, p.v_scale[p.per_head ? g : 0],
                                             reinterpret_cast<float*>(sK));
}

template <int D, int G>
cudaError_t launch_decode_tc_t(const DecodeParams& p, cudaStream_t s) {
  using C = DecodeTcCfg<D, G>;
  if (p.bps > C::MAX_BPS || p.bps % C::TPB != 0) return cudaErrorInvalidValue;  // whole tiles
  CUtensorMap tmk, tmv;
  if (!make_pool_map(&tmk, const_cast<uint8_t*>(p.k_cache), D, p.Hkv, p.num_blocks, C::RB) ||
      !make_pool_map(&tmv, const_cast<uint8_t*>(p.v_cache), D, p.Hkv, p.num_blocks, C::RB))
    return cudaErrorInvalidValue;
  auto kern = decode_tc_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_splits, p.Hkv, p.B);
  return launch_dependent(kern, grid, dim3(kDecodeTcThreads), C::SMEM, s, p, tmk, tmv);
}

template <int D>
cudaError_t launch_decode_tc_g(const DecodeParams& p, int G, cudaStream_t s) {
  switch (G) {
    case 1: return launch_decode_tc_t<D, 1>(p, s);
    case 2: return launch_decode_tc_t<D, 2>(p, s);
    case 4: return launch_decode_tc_t<D, 4>(p, s);
    case 8: return launch_decode_tc_t<D, 8>(p, s);
    case 16: return launch_decode_tc_t<D, 16>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_uses_tensor_cores(int D, int elt) { return elt == 1 && (D == 64 || D == 128 || D == 256); }

cudaError_t launch_decode_tc(const DecodeParams& p, int D, int G, cudaStream_t s) {
  if (D == 64) return launch_decode_tc_g<64>(p, G, s);
  if (D == 128) return launch_decode_tc_g<128>(p, G, s);
  if (D == 256) return launch_decode_tc_g<256>(p, G, s);
  return cudaErrorInvalidValue;
}

}  // namespace fkv
