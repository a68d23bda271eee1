// FP8 prefill (chunked) attention on tcgen05 tensor cores, two-level accumulation.
//
// The vLLM blog "FP8 KV-Cache and Attention quantization in vLLM": with an FP8 KV cache
// the whole attention runs in FP8, the QK and the Score*V matrix products included
// (引言); FP8 tensor cores accumulate imprecisely over long contractions, so each partial
// accumulation is promoted into a true FP32 register (section "Kernel 与 vLLM 改进",
// paragraph "Two-level accumulation"); head_dim 256 puts the most pressure on that
// scheme (section "大 Head Dimension 的限制").
//
// CTA = (128-query tile, query head h, sequence b); 16 warps (12 on bf16 layers; one fewer
// on bf16 layers at head_dim 256):
//   warps 0-7  softmax: quantise the Q tile to e4m3 into shared memory (bf16 layers copy
//              it); then per key tile warp w owns 16 query rows of its SM quarter (TMEM
//              lanes 32 (w % 4) + 16 (w / 4) ..), lanes l and l + 16 each half of a row's
//              columns (16x32bx2 TMEM loads): scale, mask (causal, sliding window), the row
//              maximum (one shuffle between the halves), online softmax (running max m,
//              unrounded sum l per half), write P8 = e4m3(p * 448) (bf16 layers: P rounded
//              to bf16) into shared memory, publish the tile's alpha.  Two softmax warps
//              per SM quarter hide each other's TMEM and barrier latency.  (bf16 layers:
//              warps 0-3, one whole row per lane.)
//   next 4     correction warpgroup: promote the tile's P.V partial from TMEM into the
//              FP32 accumulator O = O * alpha + O_tile (every tile, every N tiles, or
//              never); epilogue O * v_s / l -> bf16 (l sums p * 448 on e4m3 layers).  On
//              e4m3 layers O is held in these threads' registers (one row per thread; at
//              head_dim 256 its first 128 columns, the rest in TMEM).
//   next       TMA, K tiles: each 16-token block is one box [16][row bytes] of the paged
//              pool (4-D tensor map: row bytes, slot-in-block, KV head, block).
//   next       allocates TMEM, issues S = Q8 K8^T with tcgen05.mma (kind::f8f6f4 for e4m3,
//              kind::f16 for bf16; FP32 accumulation in TMEM), commits to mbarriers.
//   next       issues O_tile = P8 V8 the same way (an MMA issue holds its thread for about
//              the product's duration, so the two chains run on two warps).
//   last       TMA, V tiles (a warp's copies go out one after another, so K and V have a
//              warp each, except bf16 layers at head_dim 256, where the K warp copies
//              both).
// Key tiles hold 128 keys (64 for bf16 head_dim 256).  TMEM columns, by instantiation:
//   e4m3 up to head_dim 128: two S buffers [0, 256), two O_tile buffers from 256; O in the
//     correction warps' registers (with promote_every 0 the tensor core accumulates into
//     O_tile buffer 0).  The QK^T of tile t+1 then runs while the softmax works on tile t,
//     and the P.V of tile t while tile t-1 is promoted.  The registers come from
//     per-warpgroup budgets (setmaxnreg): softmax 120, correction 232, copy and MMA warps
//     40 per thread.  Windowed layers write P8 back into TMEM over the S columns each
//     thread has read, and P.V takes it from there as its A operand;
//   e4m3 at head_dim 256 (full or windowed): one S buffer [0, 128), two 128-column O_tile
//     buffers [128, 384) that take the two N = 128 halves of each P.V product, and the
//     second half of O at [384, 512); the first half of O in registers.  Each half is
//     promoted while the tensor core works on the other.  With promote_every >= 2 or 0
//     the running sum spans both O_tile buffers;
//   bf16 layers: one S buffer [0, 128), O_tile (two buffers up to head_dim 128), O in
//     TMEM; at head_dim 256 the P.V product runs as two N = 128 halves through one O_tile.
// Every wait is bounded in time; a timeout records FKV_FAULT_TIMEOUT, lets the CTA's
// copies and MMAs drain and returns.
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace fkv {

constexpr float kLog2E4m3Max = 8.807354922057604f;  // log2(448)

FKV_DEV float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum of N values as a tree of three-input maxima (depth log3 N, rather than a chain
// of N / 2 dependent operations).
template <int N>
FKV_DEV float max_tree(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else if constexpr (N == 2) {
    return fmaxf(v[0], v[1]);
  } else {
    constexpr int A = (N + 2) / 3, B = (N - A + 1) / 2;
    return fmax3(max_tree<A>(v), max_tree<B>(v + A), max_tree<N - A - B>(v + A + B));
  }
}

// The waits of this kernel take their timed path inline: the warpgroups of the e4m3
// instantiations up to head_dim 128 run under different register budgets, which one
// out-of-line function cannot serve (and inline waits measured faster at head_dim 256 too).
FKV_DEV bool pf_wait(uint64_t* bar, uint32_t parity) { return wait_ns<true>(bar, parity); }
FKV_DEV bool pf_wait_warp(uint64_t* bar, uint32_t parity) { return wait_warp<true>(bar, parity); }

// An empty statement that "uses and redefines" 32 values: placed after the arithmetic on them,
// it keeps the compiler from moving that arithmetic below the next TMEM load (which would
// keep every chunk's loaded values live at once).
FKV_DEV void pin32(float* v) {
  asm volatile("" : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]), "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]), "+f"(v[30]), "+f"(v[31]));
}

template <int D, bool BF, bool WIN>
struct PrefillCfg {
  static constexpr int ES = BF ? 2 : 1;             // bytes per element (bf16 / e4m3)
  // 128 queries per CTA; 128 keys per tile, or 64 for bf16 head_dim 256, whose 128-key
  // K and V tiles would not fit next to the Q tile in shared memory
  static constexpr int BM = 128, BN = (BF && D > 128) ? 64 : 128;
  static constexpr int NBLK = BN / 16;              // 16-token pool blocks per key tile
  static constexpr int NCH = BN / 32;               // 32-column chunks of an S row
  static constexpr int DB = D * ES;                 // bytes of one Q / K / V row
  static constexpr int RB = DB < 128 ? DB : 128;    // bytes of one swizzled row
  static constexpr int NSUB = DB / RB;              // sub-tiles along head_dim
  static constexpr int EPS = RB / ES;               // elements of a sub-tile row: N of one P.V product
  static constexpr int SWZ = RB == 128 ? 2 : 4;     // descriptor swizzle mode (128 B / 64 B)
  static constexpr int SUB = BM * RB;               // bytes of one 128-row Q sub-tile
  static constexpr int TILE = BM * DB;              // bytes of the Q tile
  static constexpr int KSUB = BN * RB;              // bytes of one BN-row K / V sub-tile
  static constexpr int KTILE = BN * DB;             // bytes of a K or V tile
  static constexpr int NS = (!BF && D <= 128) ? 3 : 2;  // K/V stages
  static constexpr int DN = D < 128 ? D : 128;      // O_tile width (elements) of one P.V pass
  static constexpr int NH = D / DN;                 // P.V passes
  static constexpr int PB = BN * ES;                // bytes of one P row
  static constexpr int PTILE = BM * PB;             // bytes of one P tile
  static constexpr int KSTEP = 32 / ES;             // keys (P columns) of one P.V k-step (32 bytes)
  // Windowed e4m3 up to head_dim 128: each thread writes its P8 back into TMEM over the S
  // columns it has read, and P.V takes P8 from there as its A operand (measured 3 % faster
  // there; with full attention, no faster).  Otherwise P goes through shared memory.
  static constexpr bool TS = !BF && D <= 128 && WIN;
  // e4m3 layers: the FP32 accumulator O lives in the correction warps' registers (at
  // head_dim 256 its first half), which take registers from the other warpgroups through
  // setmaxnreg; the freed TMEM holds two O_tile buffers (and two S buffers up to head_dim
  // 128, where windowed layers also keep P8 in them).
  static constexpr bool REGO = !BF;
  static constexpr int SBUF = (TS || (REGO && D <= 128)) ? 2 : 1;  // S buffers in TMEM
  static constexpr int OTB = (REGO || (!TS && D <= 128)) ? 2 : 1;  // O_tile buffers in TMEM
  // unrolling of the softmax / correction chunk loops: full for head_dim <= 128 (the
  // softmax is the critical path there), none for 256 (code size of four warp roles)
  static constexpr int UNR = D <= 128 ? 4 : 1;
  static constexpr bool ONE_LOAD = D <= 128 || !BF;  // S row loaded once into registers
  // e4m3 layers up to head_dim 128 mask a partly visible tile by setting its hidden scores
  // to -inf in registers (one code path for every tile); head_dim 256 keeps a masked copy
  // of the exponent pass, which measured slightly faster there
  static constexpr bool PREMASK = !BF && D <= 128;
  // the softmax tests its P and alpha slots without blocking as soon as S arrives (and
  // waits later only if they were not free); full attention at head_dim 256 measured
  // faster waiting for them only where they are written
  static constexpr bool PRETEST = D <= 128 || WIN;
  // full attention at head_dim 256 waits for S(t+1) and issues its loads right after
  // publishing P8(t), ahead of tile t's alpha (measured 0.5 % faster there; up to head_dim
  // 128 the same order was slower)
  static constexpr bool PIPE = D == 256 && !BF && !WIN;
  // softmax warps per S row: two on e4m3 layers (each half of the row's columns, so that
  // every SM quarter has two softmax warps to switch between); one on bf16 layers, whose
  // 2-byte tiles leave no shared memory for the half-row exchange
  static constexpr int SPLIT = BF ? 1 : 2;
  static constexpr int HC = BN / SPLIT;             // columns of a softmax thread
  static constexpr int HCH = HC / 32;               // its 32-column chunks
  static constexpr int SW = 4 * SPLIT;              // softmax warps (then 4 correction, K copies, 2 MMA, V copies)
  // TMA warps: K and V apart, except on bf16 layers at head_dim 256, whose kernel (two boxes
  // per block, two stages) measured faster with one warp copying both
  static constexpr int KVW = (D <= 128 || REGO) ? 2 : 1;
  static constexpr int THREADS = 32 * (SW + 6 + KVW);
  // TMEM columns; with REGO, "O" in TMEM is O_tile buffer 0 (used only when the tensor
  // core accumulates the whole contraction, promote_every 0)
  static constexpr int TM_OT = 128 * SBUF, TM_OA = REGO ? TM_OT : TM_OT + OTB * DN;
  // REGO: O columns [0, DR) in registers, [DR, D) (head_dim 256) in TMEM from TM_OH
  static constexpr int DR = REGO ? DN : 1, TM_OH = TM_OT + OTB * DN;
  static constexpr int TM_COLS = (TM_OT + OTB * DN + (REGO ? D - DN : D)) <= 256 ? 256 : 512;
  // register budgets per warpgroup with REGO (launch: 128 per thread, 512 threads): softmax
  // warpgroups 120, the correction warpgroup 232 (144 at head_dim 64), the copy / MMA
  // warpgroup the rest.  setmaxnreg.dec may only lower and .inc only raise a budget.
  static constexpr int REG_LAUNCH = 128, REG_SOFT = 120, REG_CORR = D > 64 ? 232 : 144,
                       REG_MISC = 4 * REG_LAUNCH - 2 * REG_SOFT - REG_CORR;
  // shared memory layout (bytes)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NS * KTILE;
  static constexpr int OFF_P = OFF_V + NS * KTILE;          // two P tiles
  static constexpr int OFF_A = OFF_P + 2 * PTILE;           // alpha [2][128] floats
  static constexpr int OFF_L = OFF_A + 2 * BM * 4;          // l [SPLIT][128] floats
  static constexpr int OFF_BAR = OFF_L + SPLIT * BM * 4;
  static constexpr int NBAR = 19 + 4 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t IDESC_QK = BF ? idesc_bf16_f32(128, BN, 0, 0) : idesc_e4m3_f32(128, BN, 0, 0);
  static constexpr uint32_t IDESC_PV = BF ? idesc_bf16_f32(128, EPS, 0, 1) : idesc_e4m3_f32(128, EPS, 0, 1);
  static_assert(TM_OA + D <= 512 && TM_OT + OTB * DN <= 512 && (!REGO || TM_OH + D - DN <= 512), "TMEM budget");
  static_assert(!REGO || (THREADS == 512 && 2 * REG_SOFT + REG_CORR + REG_MISC <= 4 * REG_LAUNCH),
                "register budgets of the warpgroups");
  static_assert(!REGO || (REG_SOFT <= REG_LAUNCH && REG_MISC <= REG_LAUNCH && REG_CORR >= REG_LAUNCH),
                "budgets lowered by setmaxnreg.dec and raised by .inc");
  static_assert(!REGO || (REG_SOFT % 8 == 0 && REG_CORR % 8 == 0 && REG_MISC % 8 == 0 && REG_MISC >= 24 &&
                          REG_CORR <= 256),
                "setmaxnreg counts: multiples of 8 in [24, 256]");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(!ONE_LOAD || BN == 128, "the one-load softmax holds a 128-column S row");
  static_assert(HC % 32 == 0 && (HCH % 2 == 0 || ONE_LOAD || HCH == 1), "softmax chunks");
  static_assert(!TS || (SPLIT == 2 && ONE_LOAD && HC == 64), "P8 in TMEM: 64 columns (16 words) per thread");
};

// One MMA of the element type: e4m3 (kind::f8f6f4) or bf16 (kind::f16), FP32 accumulation.
template <bool BF>
FKV_DEV void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  if constexpr (BF) umma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
  else umma_f8(d_tmem, adesc, bdesc, idesc, accumulate);
}

template <int D, bool BF, bool WIN>
__global__ void __launch_bounds__(PrefillCfg<D, BF, WIN>::THREADS, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  using C = PrefillCfg<D, BF, WIN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;
  float* sAlpha = reinterpret_cast<float*>(smem + C::OFF_A);
  float* sL = reinterpret_cast<float*>(smem + C::OFF_L);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;      // [2]
  uint64_t* s_free = bars + 3;      // [2]
  uint64_t* p_full = bars + 5;      // [2]
  uint64_t* p_free = bars + 7;      // [2]
  uint64_t* o_full = bars + 9;      // [2] O_tile of P.V pass n in buffer n % OTB
  uint64_t* o_free = bars + 11;     // [2]
  uint64_t* l_full = bars + 13;
  uint64_t* mma_done = bars + 14;
  uint64_t* a_full = bars + 15;     // [2] alpha of a tile published in slot t % 2
  uint64_t* a_free = bars + 17;     // [2] ... and read by the correction warpgroup
  uint64_t* k_full = bars + 19;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* v_full = k_empty + C::NS;
  uint64_t* v_empty = v_full + C::NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = gridDim.x - 1 - blockIdx.x;  // longest (latest) query tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int G = p.Hq / p.Hkv;
  const int g = h / G;

  // ------------------------------------------------------------ sequence geometry
  const int r0 = p.cu_q[b];
  const int Lq = p.cu_q[b + 1] - r0;
  int T = p.context_lens[b];
  if (T < 0 || T > p.max_blocks * 16) {
    if (qt == 0 && h == 0 && threadIdx.x == 0) raise_fault(p.fault, FKV_FAULT_CONTEXT);
    T = T < 0 ? 0 : p.max_blocks * 16;
  }
  if (Lq > T || Lq < 0) {
    if (qt == 0 && h == 0 && threadIdx.x == 0) raise_fault(p.fault, FKV_FAULT_QLEN);
    return;
  }
  const int q0 = qt * C::BM;  // first row of the tile within the sequence
  if (q0 >= Lq) return;
  const int rows = min(C::BM, Lq - q0);
  const int pos0 = T - Lq + q0;  // absolute position of the tile's first query
  const int kv_end = p.causal ? min(T, pos0 + rows) : T;  // keys [kv_lo, kv_end) matter
  const int kv_lo = WIN ? max(0, pos0 - p.window + 1) : 0;
  const int tb = kv_lo / C::BN;                               // first key tile
  const int n_t = (kv_end + C::BN - 1) / C::BN - tb;          // tiles u = 0 .. n_t-1 are tb + u
  const int nblk_seq = (T + 15) >> 4;

  // barriers signalled by the softmax or correction warps count warps (one arrival each)
  constexpr int NSM = C::SW;  // softmax warps
  if (threadIdx.x == 0) {
    mbar_init(q_full, NSM);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], C::TS ? 1 : NSM);  // TS: released by the P.V that read P8 from it
      mbar_init(&p_full[i], NSM);
      mbar_init(&p_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], NSM);
      mbar_init(&a_free[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 4);
    }
    mbar_init(l_full, NSM);
    mbar_init(mma_done, 2);  // one commit from each MMA warp
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    *abort_s = 0;
    fence_mbar_init();
  }
  if (warp == C::SW + 5) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < C::SW) {
    // ============================================================ softmax warps
    if constexpr (C::REGO && C::REG_SOFT < C::REG_LAUNCH) regs_dec<C::REG_SOFT>();
    // SPLIT 1: warp w holds the 32 rows of its SM quarter (TMEM lanes 32 (w % 4) ..), one per
    // lane, all columns.  SPLIT 2: warp w holds 16 of them, 32 (w % 4) + 16 (w / 4) + (lane % 16),
    // lanes l and l + 16 each half of the row's columns (the 16x32bx2 TMEM load shape), so that
    // the row maximum is one shuffle away.
    const int hf = C::SPLIT == 2 ? lane >> 4 : 0;  // column half
    const int rb = C::SPLIT == 2 ? (warp & 3) * 32 + (warp >> 2) * 16 : (warp & 3) * 32;  // first TMEM lane
    const int i = rb + (C::SPLIT == 2 ? (lane & 15) : lane);  // query row within the tile (TMEM lane i)
    const bool row_ok = i < rows;
    const int pos = pos0 + i;                  // its absolute position
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(rb) << 16);
    const int c0 = hf * C::HC;                 // first column of this thread's half
    // ---- prologue: Q row -> e4m3 codes (bf16 values on bf16 layers) in the swizzled Q tile;
    // the row's 16-byte chunks are shared between the row's SPLIT threads
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(r0 + q0 + i) * p.Hq + h) * D);
      const float iq = BF ? 1.f : __frcp_rn(p.q_scale[p.per_head ? h : 0]);
      constexpr int QCH = C::DB / 16 / C::SPLIT;  // chunks per thread
#pragma unroll 4
      for (int cc = 0; cc < QCH; ++cc) {
        const int c = hf * QCH + cc;
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (row_ok) {
          if constexpr (BF) {
            out = src[c];
          } else {
            const uint4 a = src[2 * c], bq = src[2 * c + 1];
            const uint32_t in[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 x0 = bf16x2_to_f2(in[2 * j]), x1 = bf16x2_to_f2(in[2 * j + 1]);
              const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(x0.x, iq), __fmul_rn(x0.y, iq));
              const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(x1.x, iq), __fmul_rn(x1.y, iq));
              w[j] = lo | (hi << 16);
            }
            out = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        const int byte = c * 16;
        const int sub = byte / C::RB;
        const uint32_t lin = static_cast<uint32_t>(i * C::RB + (byte % C::RB));
        *reinterpret_cast<uint4*>(sQ + sub * C::SUB + swz(lin, C::RB)) = out;
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(q_full);
    }
    const float cst = BF ? p.sm_scale_log2
                         : p.sm_scale_log2 * p.q_scale[p.per_head ? h : 0] * p.k_scale[p.per_head ? g : 0];
    const int lim_row = (p.causal && row_ok) ? min(T, pos + 1) : T;  // keys [lo_row, lim_row) visible
    const int lo_row = (WIN && row_ok) ? max(0, pos - p.window + 1) : 0;
    float m = -INFINITY, l = 0.f;              // l: this thread's columns only
    bool ok = true;
    // the half row of S in registers (one-load softmax)
    float vall[C::ONE_LOAD ? C::HC : 1];
    // PIPE: wait for S(t) and issue the loads of this thread's half row (called before the
    // loop for tile 0 and at the end of tile t-1 for tile t)
    auto load_s_row = [&](int t) -> bool {
      const int sb = t % C::SBUF;
      if (!pf_wait_warp(&s_full[sb], (t / C::SBUF) & 1)) return false;
      tc_fence_after();
      if constexpr (C::PIPE) {
        const uint32_t sc = lane_base + 128 * sb;
#pragma unroll
        for (int c = 0; c < C::HCH; ++c) tmem_ld32_16x2<C::HC>(sc + 32 * c, *reinterpret_cast<float(*)[32]>(vall + 32 * c));
      }
      return true;
    };
    if constexpr (C::PIPE) ok = n_t == 0 || load_s_row(0);
    for (int t = 0; ok && t < n_t; ++t) {
      // another warp's timeout is noticed every 8 tiles (every wait is bounded anyway)
      if ((t & 7) == 7 && abort_warp(abort_s)) { ok = false; break; }
      const int sb = t % C::SBUF;
      if constexpr (!C::PIPE) {
        if (!pf_wait_warp(&s_full[sb], (t / C::SBUF) & 1)) { ok = false; break; }
        tc_fence_after();
      }
      // chunk c (32 columns) of this thread's columns: its own 32 columns of the row from
      // [c0 + 32 c, ...), where the 16x32bx2 shape adds c0 = HC for the upper lanes itself
      const uint32_t sc = lane_base + 128 * sb;
      auto ld_s = [&](int c, float (&v)[32]) {
        if constexpr (C::SPLIT == 2) tmem_ld32_16x2<C::HC>(sc + 32 * c, v);
        else tmem_ld32(sc + 32 * c, v);
      };
      // one-load softmax: the half row's loads go out first (with PIPE they went out at the
      // end of the previous tile); the tile's bookkeeping below runs while they are in flight
      if constexpr (C::ONE_LOAD && !C::PIPE) {
#pragma unroll
        for (int c = 0; c < C::HCH; ++c) ld_s(c, *reinterpret_cast<float(*)[32]>(vall + 32 * c));
      }
      // the P and alpha slots of tile t (freed by tile t-2's P.V and correction) are
      // normally free long before they are written: test them now without blocking, and
      // wait further down only if they were not
      const int pb = t & 1;
      const bool p_ready = C::TS || t < 2 || (C::PRETEST && mbar_test_wait(&p_free[pb], ((t >> 1) - 1) & 1));
      const bool a_ready = t < 2 || (C::PRETEST && mbar_test_wait(&a_free[pb], ((t >> 1) - 1) & 1));
      const int kbase = (tb + t) * C::BN + c0;  // key of this thread's first column
      const int lim = lim_row - kbase;      // columns [lo, lim) of this thread's half are visible
      // full-attention instantiations fold the lower bound away (it costs the softmax
      // warps dearly when it is a run-time value)
      const int lo = WIN ? lo_row - kbase : -(1 << 30);
      const bool full = lim >= C::HC && (!WIN || lo <= 0);  // nothing masked in this half
      // nothing masked in any row of the warp: selects the unmasked code paths, which hold
      // warp-collective TMEM loads and so must be taken by the whole warp (a masked path
      // is correct for every row)
      const bool wfull = __all_sync(0xffffffffu, full);
      float tmax = -INFINITY;
      if constexpr (C::ONE_LOAD) {
        // the half row in registers, one TMEM wait; S is released at once
        tmem_ld_wait();
        if constexpr (!C::TS) {  // (TS: S is freed by the P.V that reads P8 from it)
          tc_fence_before();
          mbar_arrive_warp(&s_free[sb]);
        }
        if constexpr (C::PREMASK) {
          // a warp with a partly visible row: the hidden scores of its rows become -inf
          // here, so that one unmasked code path serves every tile (2^(-inf) = 0 is their
          // p, the zero the mask asks for; cst > 0, so the maximum of the visible raw
          // scores scales to the maximum of the scaled ones).  The branch is taken by the
          // whole warp: a per-thread branch here cost the full tiles about 4 %.
          if (!wfull) {
#pragma unroll
            for (int j = 0; j < C::HC; ++j)
              if (j >= lim || j < lo) vall[j] = -INFINITY;
          }
          tmax = max_tree<C::HC>(vall) * cst;
        } else if (full) {
          tmax = max_tree<C::HC>(vall) * cst;
        } else {
#pragma unroll
          for (int j = 0; j < C::HC; ++j) tmax = fmaxf(tmax, (j < lim && j >= lo) ? vall[j] * cst : -INFINITY);
        }
      } else {
        // pass 1: max of the scaled, masked scores (cst > 0, so the raw maximum scales).
        // The TMEM loads are warp-collective: every lane issues them; only the arithmetic
        // depends on the row's own mask.
        // (the mask test is taken once per tile: tested per element, it costs every
        // element of every tile a compare and a select)
        if (wfull) {
          float mx = -INFINITY;
  #pragma unroll C::UNR
          for (int c = 0; c < C::HCH; ++c) {
            float v[32];
            ld_s(c, v);
            tmem_ld_wait();
            mx = fmaxf(mx, max_tree<32>(v));
          }
          tmax = mx * cst;
        } else {
  #pragma unroll C::UNR
          for (int c = 0; c < C::HCH; ++c) {
            float v[32];
            ld_s(c, v);
            tmem_ld_wait();
  #pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = 32 * c + j;
              tmax = fmaxf(tmax, (col < lim && col >= lo) ? v[j] * cst : -INFINITY);
            }
          }
        }
      }
      // the row's maximum: this half's and the other half's (lane l ^ 16)
      if constexpr (C::SPLIT == 2) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      const float mn = fmaxf(m, tmax);
      const float alpha = (m == -INFINITY) ? 0.f : ex2(m - mn);
      const float msafe = (mn == -INFINITY) ? 0.f : mn;
      // P tile t%2 is free once the P.V of tile t-2 completed
      if (!C::TS && !__all_sync(0xffffffffu, p_ready) && !pf_wait_warp(&p_free[pb], ((t >> 1) - 1) & 1)) { ok = false; break; }
      uint8_t* P = sP + pb * C::PTILE;
      // pass 2: p = 2^(s*cst - m), its unrounded sum, and P8 = e4m3(p * 448) into the P tile;
      // the next chunk's TMEM load is in flight while the current one is processed
      float2 lsum2 = make_float2(0.f, 0.f);
      // e4m3 layers fold the factor 448 of P8 into the exponent: p * 448 = 2^(s*cst - m + log2 448),
      // so l sums p * 448 and the epilogue divides by l alone
      const float nb = (BF ? 0.f : kLog2E4m3Max) - msafe;
      const float2 cst2 = make_float2(cst, cst), nm2 = make_float2(nb, nb);
      uint32_t ptm[C::TS ? 2 * C::HCH * 4 : 1];  // TS: this thread's P8 words (four keys each)
      // c: chunk of this thread's half; `masked` says whether to apply the row's mask, which
      // only tiles not wholly visible need: never on e4m3 layers up to head_dim 128 (the
      // hidden scores are -inf already), a compile-time flag at head_dim 256 (the choice is
      // made once per tile), the run-time test of `full` on bf16 layers (whose registers do
      // not hold two copies of the loop)
      auto chunk = [&](const float (&v)[32], int c, auto masked) {
        constexpr int MASKED = decltype(masked)::value;  // 0 never, 1 always, 2 unless full
        uint32_t pk[8 * C::ES];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float2 x0 = __ffma2_rn(make_float2(v[j], v[j + 1]), cst2, nm2);
          float2 x1 = __ffma2_rn(make_float2(v[j + 2], v[j + 3]), cst2, nm2);
          x0.x = ex2(x0.x); x0.y = ex2(x0.y); x1.x = ex2(x1.x); x1.y = ex2(x1.y);
          if (MASKED == 1 || (MASKED == 2 && !full)) {
            const int col = 32 * c + j;
            if (col >= lim || col < lo) x0.x = 0.f;
            if (col + 1 >= lim || col + 1 < lo) x0.y = 0.f;
            if (col + 2 >= lim || col + 2 < lo) x1.x = 0.f;
            if (col + 3 >= lim || col + 3 < lo) x1.y = 0.f;
          }
          lsum2 = __fadd2_rn(lsum2, __fadd2_rn(x0, x1));
          if constexpr (BF) {
            __nv_bfloat162 b0 = __floats2bfloat162_rn(x0.x, x0.y), b1 = __floats2bfloat162_rn(x1.x, x1.y);
            pk[j / 2] = *reinterpret_cast<uint32_t*>(&b0);
            pk[j / 2 + 1] = *reinterpret_cast<uint32_t*>(&b1);
          } else {
            pk[j / 4] = static_cast<uint32_t>(f32x2_to_e4m3x2(x0.x, x0.y)) |
                        (static_cast<uint32_t>(f32x2_to_e4m3x2(x1.x, x1.y)) << 16);
          }
        }
        if constexpr (C::TS) {
#pragma unroll
          for (int q = 0; q < 8; ++q) ptm[8 * c + q] = pk[q];
        } else {
          // 32 columns = 32 * ES bytes of the P row, in 16-byte pieces
#pragma unroll
          for (int q = 0; q < 2 * C::ES; ++q) {
            const int byte = (c0 + 32 * c) * C::ES + 16 * q;
            const uint32_t lin = static_cast<uint32_t>(i * 128 + (byte % 128));
            *reinterpret_cast<uint4*>(P + (byte / 128) * (C::BM * 128) + swz(lin, 128)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      };
      using Unmasked = std::integral_constant<int, 0>;
      using Masked = std::integral_constant<int, 1>;
      using MaskedUnlessFull = std::integral_constant<int, 2>;
      // the whole pass 2 for one masking mode
      auto pass2 = [&](auto masked) {
        if constexpr (C::ONE_LOAD) {
#pragma unroll
          for (int c = 0; c < C::HCH; ++c) chunk(*reinterpret_cast<const float(*)[32]>(vall + 32 * c), c, masked);
        } else if constexpr (C::HCH == 1) {
          float va[32];
          ld_s(0, va);
          tmem_ld_wait();
          chunk(va, 0, masked);
        } else {
          float va[32], vb[32];
          ld_s(0, va);
    #pragma unroll C::UNR
          for (int c = 0; c < C::HCH; c += 2) {
            tmem_ld_wait();
            ld_s(c + 1, vb);
            chunk(va, c, masked);
            tmem_ld_wait();
            if (c + 2 < C::HCH) ld_s(c + 2, va);
            chunk(vb, c + 1, masked);
          }
        }
      };
      if constexpr (BF) {
        pass2(MaskedUnlessFull());
      } else if constexpr (C::PREMASK) {
        pass2(Unmasked());  // hidden scores are -inf already
      } else {
        if (wfull) pass2(Unmasked());
        else pass2(Masked());
      }
      if constexpr (C::ONE_LOAD) {
        if constexpr (C::TS) {
          // P8 over the first 16 of this thread's S columns (already read): keys 4w .. 4w+3
          // of its half in column c0 + w of S buffer sb
          tmem_st16_16x2<C::HC>(sc, ptm);
          tmem_st_wait();
        }
      }
      if constexpr (C::PIPE) {
        fence_proxy_async_smem();
        mbar_arrive_warp(&p_full[pb]);
        if (t + 1 < n_t && !load_s_row(t + 1)) { ok = false; break; }
      }
      const float lsum = lsum2.x + lsum2.y;
      if constexpr (!C::ONE_LOAD) {
        tc_fence_before();
        mbar_arrive_warp(&s_free[sb]);
      }
      l = l * alpha + lsum;
      m = mn;
      // alpha (the same in both halves) is written by half 0; its slot t%2 is free once the
      // correction warpgroup has read tile t-2's alpha
      if (!__all_sync(0xffffffffu, a_ready) && !pf_wait_warp(&a_free[pb], ((t >> 1) - 1) & 1)) { ok = false; break; }
      if (hf == 0) sAlpha[pb * C::BM + i] = alpha;
      mbar_arrive_warp(&a_full[pb]);
      if constexpr (!C::PIPE) {
        if constexpr (C::TS) tc_fence_before();
        else fence_proxy_async_smem();
        mbar_arrive_warp(&p_full[pb]);
      }
    }
    if constexpr (C::PIPE) tmem_ld_wait();  // no load left in flight on an early exit
    if (!ok) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      *abort_s = 1;
    }
    sL[hf * C::BM + i] = l;
    mbar_arrive_warp(l_full);
  } else if (warp < C::SW + 4) {
    // ============================================================ correction warpgroup
    if constexpr (C::REGO) regs_inc<C::REG_CORR>();  // O in registers
    const int i = threadIdx.x - 32 * C::SW;    // query row (TMEM lane i)
    const bool row_ok = i < rows;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp - C::SW) * 32) << 16);
    int npv = 0;
    bool ok = true;
    const int pe = p.promote_every;
    // REGO: the FP32 accumulator O of this row: columns [0, DR) in registers, the rest
    // (head_dim 256) in TMEM at TM_OH
    float O[C::DR];
#pragma unroll
    for (int j = 0; j < C::DR; ++j) O[j] = 0.f;
    // the promotion of one O_tile pass into O: hn 0 into the registers, hn 1 into TMEM
    // (first: O takes the partial itself)
    auto promote_pass = [&](uint32_t src, int hn, float alpha, auto first) {
      if (hn == 0) {
        // two 32-column loads per TMEM wait (one at head_dim 64, whose correction warps
        // run under a smaller register budget)
        constexpr int PAIR = (D >= 128 && (C::DN / 32) % 2 == 0) ? 2 : 1;
#pragma unroll
        for (int c2 = 0; c2 < C::DN / 32; c2 += PAIR) {
          float ot[PAIR][32];
#pragma unroll
          for (int u = 0; u < PAIR; ++u) tmem_ld32(src + 32 * (c2 + u), ot[u]);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < PAIR; ++u) {
            const int c = c2 + u;
            if constexpr (decltype(first)::value) {
#pragma unroll
              for (int j = 0; j < 32; ++j) O[32 * c + j] = ot[u][j];
            } else {
              // packed: two fused multiply-adds per instruction, the same rounding as fmaf
              const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const float2 r = __ffma2_rn(make_float2(O[32 * c + j], O[32 * c + j + 1]), a2,
                                            make_float2(ot[u][j], ot[u][j + 1]));
                O[32 * c + j] = r.x;
                O[32 * c + j + 1] = r.y;
              }
            }
            pin32(O + 32 * c);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < C::DN / 32; ++c) {
          float ot[32], oh[32];
          const uint32_t dst = lane_base + C::TM_OH + (hn - 1) * C::DN + 32 * c;
          tmem_ld32(src + 32 * c, ot);
          if constexpr (!decltype(first)::value) tmem_ld32(dst, oh);
          tmem_ld_wait();
          if constexpr (decltype(first)::value) {
#pragma unroll
            for (int j = 0; j < 32; ++j) oh[j] = ot[j];
          } else {
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float2 r = __ffma2_rn(make_float2(oh[j], oh[j + 1]), a2, make_float2(ot[j], ot[j + 1]));
              oh[j] = r.x;
              oh[j + 1] = r.y;
            }
          }
          tmem_st32(dst, oh);
        }
        tmem_st_wait();
      }
    };
    if constexpr (C::REGO) {
      if (pe == 1) {
        // two-level accumulation every tile: O = O * alpha + O_tile(t); pass hn of tile t is
        // P.V product NH t + hn, in O_tile buffer (NH t + hn) % 2 (tile 0 assigns O: a
        // select per element instead costs the register allocation dearly)
        auto promote = [&](int t, auto first) -> bool {
          if (!pf_wait_warp(&a_full[t & 1], (t >> 1) & 1)) return false;
          const float alpha = sAlpha[(t & 1) * C::BM + i];
          mbar_arrive_warp(&a_free[t & 1]);
#pragma unroll
          for (int hn = 0; hn < C::NH; ++hn) {
            const int n = C::NH * t + hn, ob = n & 1;
            if (!pf_wait_warp(&o_full[ob], (n >> 1) & 1)) return false;
            tc_fence_after();
            promote_pass(lane_base + C::TM_OT + ob * C::DN, hn, alpha, first);
            tc_fence_before();
            mbar_arrive_warp(&o_free[ob]);
          }
          return true;
        };
        ok = n_t == 0 || promote(0, std::true_type());
        for (int t = 1; ok && t < n_t; ++t) {
          if ((t & 7) == 7 && abort_warp(abort_s)) { ok = false; break; }
          ok = promote(t, std::false_type());
        }
      } else {
        // the running sum over all D columns from TM_OT (O_tile buffer 0, or both buffers at
        // head_dim 256), rescaled in place when a row's maximum moved; promoted into O
        // every pe tiles (pe >= 2) or never (pe == 0: O stays in TMEM)
        float A = 1.f;
        bool first = true;
        for (int t = 0; t < n_t; ++t) {
          if ((t & 7) == 7 && abort_warp(abort_s)) { ok = false; break; }
          if (!pf_wait_warp(&a_full[t & 1], (t >> 1) & 1)) { ok = false; break; }
          const float alpha = sAlpha[(t & 1) * C::BM + i];
          mbar_arrive_warp(&a_free[t & 1]);
          A *= alpha;
          const bool start = pe == 0 ? t == 0 : (t % pe) == 0;
          if (!start) {
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) {
                float x[32];
                tmem_ld32(lane_base + C::TM_OT + 32 * c, x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] *= alpha;
                tmem_st32(lane_base + C::TM_OT + 32 * c, x);
              }
              tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive_warp(o_free);
          }
          if (!pf_wait_warp(o_full, t & 1)) { ok = false; break; }
          tc_fence_after();
          const bool last = pe != 0 && ((t + 1) % pe == 0 || t == n_t - 1);
          if (last) {
#pragma unroll
            for (int hn = 0; hn < C::NH; ++hn) {
              if (first) promote_pass(lane_base + C::TM_OT + hn * C::DN, hn, A, std::true_type());
              else promote_pass(lane_base + C::TM_OT + hn * C::DN, hn, A, std::false_type());
            }
            first = false;
            A = 1.f;
            tc_fence_before();
            mbar_arrive_warp(o_free);
          }
        }
      }
    } else if (pe == 1) {
      // two-level accumulation every tile: O = O * alpha + O_tile after each P.V
      for (int t = 0; t < n_t; ++t) {
        if ((t & 7) == 7 && abort_warp(abort_s)) { ok = false; break; }
        if (!pf_wait_warp(&a_full[t & 1], (t >> 1) & 1)) { ok = false; break; }
        const float alpha = sAlpha[(t & 1) * C::BM + i];
        mbar_arrive_warp(&a_free[t & 1]);
        for (int hn = 0; hn < C::NH; ++hn) {
          const int ob = npv % C::OTB;
          if (!pf_wait_warp(&o_full[ob], (npv / C::OTB) & 1)) { ok = false; break; }
          ++npv;
          tc_fence_after();
#pragma unroll C::UNR
          for (int c = 0; c < C::DN / 32; ++c) {
            float ot[32], oa[32];
            tmem_ld32(lane_base + C::TM_OT + ob * C::DN + 32 * c, ot);
            if (t > 0) tmem_ld32(lane_base + C::TM_OA + hn * C::DN + 32 * c, oa);
            tmem_ld_wait();
            if (t > 0) {
#pragma unroll
              for (int j = 0; j < 32; ++j) oa[j] = fmaf(oa[j], alpha, ot[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) oa[j] = ot[j];
            }
            tmem_st32(lane_base + C::TM_OA + hn * C::DN + 32 * c, oa);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(&o_free[ob]);
        }
        if (!ok) break;
      }
    } else {
      // promote every pe tiles (pe >= 2, one P.V product per tile) or never (pe == 0: the
      // tensor core accumulates the whole contraction into O).  The running sum the next
      // P.V accumulates into is rescaled in place when a row's maximum moved.
      const uint32_t acc_col = pe == 0 ? C::TM_OA : C::TM_OT;
      const int acc_cols = pe == 0 ? D : C::DN;
      float A = 1.f;         // product of the alphas since the last promotion
      bool have_o = false;   // O holds promoted groups
      for (int t = 0; t < n_t; ++t) {
        if ((t & 7) == 7 && abort_warp(abort_s)) { ok = false; break; }
        if (!pf_wait_warp(&a_full[t & 1], (t >> 1) & 1)) { ok = false; break; }
        const float alpha = sAlpha[(t & 1) * C::BM + i];
        mbar_arrive_warp(&a_free[t & 1]);
        A *= alpha;
        const bool start = pe == 0 ? t == 0 : (t % pe) == 0;
        if (!start) {
          // P.V(t-1) completed at the previous o_full wait
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < acc_cols / 32; ++c) {
              float x[32];
              tmem_ld32(lane_base + acc_col + 32 * c, x);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] *= alpha;
              tmem_st32(lane_base + acc_col + 32 * c, x);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          mbar_arrive_warp(o_free);
        }
        if (!pf_wait_warp(o_full, t & 1)) { ok = false; break; }
        tc_fence_after();
        const bool last = pe != 0 && ((t + 1) % pe == 0 || t == n_t - 1);
        if (last) {
#pragma unroll 1
          for (int c = 0; c < C::DN / 32; ++c) {
            float ot[32], oa[32];
            tmem_ld32(lane_base + C::TM_OT + 32 * c, ot);
            if (have_o) tmem_ld32(lane_base + C::TM_OA + 32 * c, oa);
            tmem_ld_wait();
            if (have_o) {
#pragma unroll
              for (int j = 0; j < 32; ++j) oa[j] = fmaf(oa[j], A, ot[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) oa[j] = ot[j];
            }
            tmem_st32(lane_base + C::TM_OA + 32 * c, oa);
          }
          tmem_st_wait();
          have_o = true;
          A = 1.f;
          tc_fence_before();
          mbar_arrive_warp(o_free);
        }
      }
    }
    if (!ok) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      *abort_s = 1;
    }
    // ---- epilogue: O * v_s / l -> bf16 (every lane loads; rows past the chunk do not store)
    if (pf_wait_warp(l_full, 0) && !abort_warp(abort_s)) {
      float l = sL[i];
      if constexpr (C::SPLIT == 2) l += sL[C::BM + i];  // the two halves' sums
      const float vs = BF ? 1.f : p.v_scale[p.per_head ? g : 0];
      const float f = (l > 0.f) ? vs / l : 0.f;  // l sums p * 448 on e4m3 layers
      __nv_bfloat16* dst = p.out + (static_cast<size_t>(r0 + q0 + i) * p.Hq + h) * D;
      // 32 values of the row, columns 32 c .. 32 c + 31, scaled and stored as bf16
      auto store32 = [&](int c, const float (&oa)[32]) {
        if (row_ok) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 y = __floats2bfloat162_rn(oa[2 * j] * f, oa[2 * j + 1] * f);
            w[j] = *reinterpret_cast<uint32_t*>(&y);
          }
          uint4* o4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int j = 0; j < 4; ++j) o4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      };
      bool from_regs = false;
      if constexpr (C::REGO) {
        if (pe != 0) {
          from_regs = true;
#pragma unroll
          for (int c = 0; c < C::DR / 32; ++c) {
            float oa[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) oa[j] = O[32 * c + j];
            store32(c, oa);
          }
#pragma unroll 1
          for (int c = C::DR / 32; c < D / 32; ++c) {
            float oa[32];
            tmem_ld32(lane_base + C::TM_OH + 32 * c - C::DR, oa);
            tmem_ld_wait();
            store32(c, oa);
          }
        }
      }
      if (!from_regs) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float oa[32];
          tmem_ld32(lane_base + C::TM_OA + 32 * c, oa);
          tmem_ld_wait();
          store32(c, oa);
        }
      }
    }
  } else {
  // the copy and MMA-issue warpgroup needs few registers
  if constexpr (C::REGO && C::REG_MISC < C::REG_LAUNCH) regs_dec<C::REG_MISC>();
  if (warp == C::SW + 4 || warp == C::SW + 7) {
    // ============================================================ TMA producers
    // Warp SW+4 copies the K tiles and warp SW+7 the V tiles: a warp's copies go out one
    // after another (about 100 cycles per 2 KiB box), so two warps halve the time a tile's
    // copies take.  On bf16 layers at head_dim 256 warp SW+4 copies both.  Lane
    // j < NBLK copies the tile's j-th 16-token block; the block ids of tile t+1 are read
    // while tile t's copies are issued.
    const int kind0 = warp == C::SW + 7 ? 1 : 0;  // 0: K, 1: V
    constexpr int KINDS = C::KVW == 2 ? 1 : 2;    // kinds this warp copies
    const int* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;
    int last[2][C::NS];  // last use of each stage whose copies were issued
#pragma unroll
    for (int s = 0; s < C::NS; ++s) last[0][s] = last[1][s] = -1;
    // blocks past the context read block 0 (their keys are masked)
    auto block_id = [&](int t) -> int {
      const int lb = (tb + t) * C::NBLK + lane;
      return (lane < C::NBLK && t < n_t && lb < nblk_seq) ? trow[lb] : 0;
    };
    int id_next = block_id(0);
    for (int t = 0; t < n_t; ++t) {
      int stop = *abort_s;
      if (lane == 0 && (t & 7) == 7 && p.fault && (*reinterpret_cast<volatile int*>(p.fault) & FKV_FAULT_TIMEOUT))
        stop = 1;  // another CTA gave up: stop early
      if (__any_sync(0xffffffffu, stop != 0)) {
        *abort_s = 1;
        break;
      }
      int id = id_next;
      if (id < 0 || id >= p.num_blocks) {
        raise_fault(p.fault, FKV_FAULT_BLOCK_ID);
        id = 0;
      }
      id_next = block_id(t + 1);
      const int st = t % C::NS, use = t / C::NS;
      bool ok = true;
#pragma unroll
      for (int kk = 0; kk < KINDS; ++kk) {
        const int kind = kind0 + kk;
        uint64_t* full = kind ? v_full : k_full;
        if (lane == 0 && use > 0) ok = pf_wait(kind ? &v_empty[st] : &k_empty[st], (use - 1) & 1);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // the expected byte count is posted before any of the copies can complete
        if (lane == 0) mbar_arrive_expect_tx(&full[st], C::KTILE);
        __syncwarp();
        if (lane < C::NBLK) {
          uint8_t* dst = (kind ? sV : sK) + st * C::KTILE + lane * 16 * C::RB;
#pragma unroll
          for (int s = 0; s < C::NSUB; ++s)
            tma_load_4d(dst + s * C::KSUB, kind ? &tmv : &tmk, s * C::RB, 0, g, id, &full[st]);
        }
        last[kind][st] = use;
      }
      if (!ok) {
        if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
        *abort_s = 1;
        break;
      }
    }
    // let every issued copy land before the CTA can exit
    if (lane == 0) {
      for (int s = 0; s < C::NS; ++s) {
        if (last[0][s] >= 0) pf_wait(&k_full[s], last[0][s] & 1);
        if (last[1][s] >= 0) pf_wait(&v_full[s], last[1][s] & 1);
      }
    }
  } else {
    // ============================================================ MMA issuers
    // Warp SW+5 issues S = Q8 K8^T, warp SW+6 O_tile = P8 V8.  A tcgen05.mma issue holds
    // its thread for about the product's execution time and a commit for tens of cycles, so
    // one thread issuing both chains (two products, five commits and five waits per tile)
    // would take longer per tile than the softmax; on two warps the chains overlap.
    const bool qk_warp = warp == C::SW + 5;
    // operand descriptors of the tile bases; every operand is one of them advanced by a
    // compile-time or per-stage byte offset (desc_add)
    const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 8 * C::RB, C::SWZ);
    const uint64_t dK = smem_desc(smem_u32(sK), 16, 8 * C::RB, C::SWZ);
    const uint64_t dV = smem_desc(smem_u32(sV), 8 * C::RB, 8 * C::RB, C::SWZ);
    const uint64_t dP = smem_desc(smem_u32(sP), 16, 1024, 2);
    int npv = 0;
    // S(t) = Q8 K8^T into S buffer t % SBUF
    auto issue_qk = [&](int t) -> bool {
      const int st = t % C::NS, sb = t % C::SBUF;
      if (!pf_wait_warp(&k_full[st], (t / C::NS) & 1)) return false;
      if (t >= C::SBUF && !pf_wait_warp(&s_free[sb], ((t / C::SBUF) - 1) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < C::DB / 32; ++kk) {
          const int byte = kk * 32;
          const uint32_t qoff = (byte / C::RB) * C::SUB + (byte % C::RB);
          const uint32_t koff = (byte / C::RB) * C::KSUB + (byte % C::RB);
          umma<BF>(tmem + 128 * sb, desc_add(dQ, qoff), desc_add(dK, st * C::KTILE + koff), C::IDESC_QK,
                   kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[sb]);
        umma_commit(&k_empty[st]);
      }
      __syncwarp();
      return true;
    };
    // One P.V pass: the DN output columns hn*DN .. of O_tile (or O) from P(t) and V(t), one
    // product of N = EPS per V sub-tile and per 32-byte k-step of P.
    auto issue_pv_pass = [&](int st, int pb, int hn, uint32_t dst, bool fresh) {
#pragma unroll
      for (int kk = 0; kk < C::PB / 32; ++kk) {
        const int pbyte = kk * 32;
        const uint64_t ad = desc_add(dP, pb * C::PTILE + (pbyte / 128) * (C::BM * 128) + (pbyte % 128));
        // TS: keys 32 kk .. of P8 sit in S buffer pb, half h = 32 kk / HC at column HC h, four
        // keys per column
        const uint32_t a_tm =
            tmem + 128 * pb + C::HC * ((32 * kk) / C::HC) + ((32 * kk) % C::HC) / 4;
#pragma unroll
        for (int j = 0; j < C::DN / C::EPS; ++j) {
          const int sub = hn * (C::DN / C::EPS) + j;
          const uint64_t bd = desc_add(dV, st * C::KTILE + sub * C::KSUB + kk * C::KSTEP * C::RB);
          const uint32_t acc = (kk > 0 || !fresh) ? 1u : 0u;
          if constexpr (C::TS) umma_f8_tmem_a(dst + j * C::EPS, a_tm, bd, C::IDESC_PV, acc);
          else umma<BF>(dst + j * C::EPS, ad, bd, C::IDESC_PV, acc);
        }
      }
    };
    // O_tile = P8(t) V8(t), in NH products of N = DN
    auto issue_pv = [&](int t) -> bool {
      const int st = t % C::NS, pb = t & 1;
      if (!pf_wait_warp(&p_full[pb], (t >> 1) & 1)) return false;
      if (!pf_wait_warp(&v_full[st], (t / C::NS) & 1)) return false;
      // keys past the context may hold stale bytes (NaN codes): zero their V rows, since
      // 0 * NaN would poison the product even though their P is 0
      const int kbase = (tb + t) * C::BN;
      if (kbase + C::BN > T) {
        const int first = max(T - kbase, 0);
        const int chunks = C::RB / 16;
        const int items = (C::BN - first) * C::NSUB * chunks;
        for (int it = lane; it < items; it += 32) {
          const int c = it % chunks;
          const int s = (it / chunks) % C::NSUB;
          const int r = first + it / (chunks * C::NSUB);
          *reinterpret_cast<uint4*>(sV + st * C::KTILE + s * C::KSUB + r * C::RB + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (p.promote_every == 1) {
        for (int hn = 0; hn < C::NH; ++hn) {
          // O_tile buffer npv % OTB is free once the correction promoted pass npv - OTB
          const int ob = npv % C::OTB;
          if (npv >= C::OTB && !pf_wait_warp(&o_free[ob], ((npv / C::OTB) - 1) & 1)) return false;
          tc_fence_after();
          if (lane == 0) issue_pv_pass(st, pb, hn, tmem + C::TM_OT + ob * C::DN, true);
          if (lane == 0) umma_commit(&o_full[ob]);
          __syncwarp();
          ++npv;
        }
      } else {
        // the running sum (O_tile, or O when never promoted) is ready once the correction
        // warpgroup has promoted or rescaled it for this tile
        if (t > 0 && !pf_wait_warp(o_free, (t - 1) & 1)) return false;
        tc_fence_after();
        const int pe = p.promote_every;
        const bool fresh = pe == 0 ? t == 0 : (t % pe) == 0;
        if (lane == 0) {
#pragma unroll
          for (int hn = 0; hn < C::NH; ++hn)
            issue_pv_pass(st, pb, hn,
                          pe == 0 ? tmem + C::TM_OA + hn * C::DN : tmem + C::TM_OT + (C::REGO ? hn * C::DN : 0),
                          fresh);
          umma_commit(o_full);
        }
        __syncwarp();
      }
      if (lane == 0) {
        umma_commit(&v_empty[st]);
        umma_commit(C::TS ? &s_free[pb] : &p_free[pb]);  // TS: P8 lived in S buffer pb
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    if (qk_warp) {
      // S(t+1) is computed while the softmax works on tile t (S is released once loaded)
      ok = pf_wait_warp(q_full, 0);
      for (int t = 0; ok && t < n_t; ++t) {
        if ((t & 7) == 7 && abort_warp(abort_s)) break;
        ok = issue_qk(t);
      }
    } else {
      for (int t = 0; ok && t < n_t; ++t) {
        if ((t & 7) == 7 && abort_warp(abort_s)) break;
        ok = issue_pv(t);
      }
    }
    if (!ok) {
      if (lane == 0) raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      *abort_s = 1;
    }
    // every MMA issued by either warp completes before TMEM is released
    if (lane == 0) {
      umma_commit(mma_done);
      pf_wait(mma_done, 0);
    }
    __syncwarp();
  }
  }
  __syncthreads();
  if (warp == C::SW + 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ------------------------------------------------------------------ host side

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

}  // namespace

// 4-D map over one pool: (D bytes, 16 slots, KV heads, blocks), box (RB bytes, 16, 1, 1).
bool make_pool_map(CUtensorMap* map, void* base, int D, int Hkv, int num_blocks, int rb) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), 16, static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(16) * D,
                                 static_cast<cuuint64_t>(16) * D * Hkv};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(rb), 16, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <int D, bool BF, bool WIN>
cudaError_t launch_prefill_t(const PrefillParams& p, void* kc, void* vc, cudaStream_t s) {
  using C = PrefillCfg<D, BF, WIN>;
  CUtensorMap tmk, tmv;
  if (!make_pool_map(&tmk, kc, C::DB, p.Hkv, p.num_blocks, C::RB) ||
      !make_pool_map(&tmv, vc, C::DB, p.Hkv, p.num_blocks, C::RB))
    return cudaErrorInvalidValue;
  auto kern = prefill_kernel<D, BF, WIN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  if constexpr (C::REGO) {
    // the warpgroups' register budgets add up to the launch's 128 per thread: a kernel built
    // with fewer would wait forever in setmaxnreg.inc, so it is never launched
    static int regs = -1;
    if (regs < 0) {
      cudaFuncAttributes a;
      e = cudaFuncGetAttributes(&a, kern);
      if (e != cudaSuccess) return e;
      regs = a.numRegs;
    }
    if (regs != C::REG_LAUNCH) return cudaErrorInvalidKernelImage;
  }
  dim3 grid(p.n_qtiles, p.Hq, p.B);
  kern<<<grid, C::THREADS, C::SMEM, s>>>(p, tmk, tmv);
  return cudaGetLastError();
}

template <int D, bool BF>
cudaError_t launch_prefill_w(const PrefillParams& p, void* kc, void* vc, cudaStream_t s) {
  return p.window > 0 ? launch_prefill_t<D, BF, true>(p, kc, vc, s) : launch_prefill_t<D, BF, false>(p, kc, vc, s);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, int D, bool bf16_layer, void* kc, void* vc, cudaStream_t s) {
  if (bf16_layer) {
    if (D == 64) return launch_prefill_w<64, true>(p, kc, vc, s);
    if (D == 128) return launch_prefill_w<128, true>(p, kc, vc, s);
    if (D == 256) return launch_prefill_w<256, true>(p, kc, vc, s);
    return cudaErrorInvalidValue;
  }
  if (D == 64) return launch_prefill_w<64, false>(p, kc, vc, s);
  if (D == 128) return launch_prefill_w<128, false>(p, kc, vc, s);
  if (D == 256) return launch_prefill_w<256, false>(p, kc, vc, s);
  return cudaErrorInvalidValue;
}

}  // namespace fkv
