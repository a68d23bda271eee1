// Paged GQA decode attention on the CUDA cores for the layers whose pools are not e4m3:
// bf16 (skip layers) and e5m2.  Split-K over the context, FP32 softmax state and P.V
// sums, then an FP32 log-sum-exp merge of the splits.  (e4m3 layers decode on the tensor
// cores, decode_tc.cu.)
//
// The vLLM blog "FP8 KV-Cache and Attention quantization in vLLM": the decode step must
// read every cached token, so its cost is the cache bytes (section "性能 Benchmark");
// skipped layers stay bf16 (section "Kernel 与 vLLM 改进", paragraph "跳过 Layer"); each
// split's partial output lives in FP32 registers and the splits are merged in FP32
// ("Two-level accumulation").  vLLM also keeps FP8 caches as e5m2 ("量子化が vLLM の推論
// 性能に与える影響", "KV キャッシュの量子化"); those codes are widened exactly to FP32 here.
//
// CTA = (split, KV head g, sequence b); it serves all G query heads of g, so each K/V
// byte is read from HBM once.  Each of the 4 warps owns two tile buffers in shared
// memory and refills one with cp.async.bulk (each 16-token block's K chunk and V chunk,
// [block][g][16][D] in the pool, completion on an mbarrier) while it computes the other;
// warp w takes tiles w, w + 4, ...  Per tile:
//   QK : lanes split (key, d-slice); FP32 FMAs; a select-free transposing shuffle
//        reduction leaves each lane with the whole score of one head;
//   softmax: running max m and sum l per head (base-2 domain), rescale factor per tile;
//   PV : lanes split (key sub-group, d-slice); acc[h][d] += p[h][key] * v[key][d].
// The warps' states are merged in shared memory and written as (o / l, log2-sum-exp).
// Every wait is bounded in time; on a timeout the CTA records FKV_FAULT_TIMEOUT, lets
// its in-flight copies land and returns.
#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"

namespace fkv {

constexpr int kNW = 4;           // warps per CTA; every warp prefetches and consumes its own tiles
constexpr int kNBUF = 2;         // tile buffers per warp (one in use, one in flight)
constexpr int kMaxBps = kMaxSplitBlocks;  // blocks per split, upper bound (table ids staged in smem)

// ELT: the pool's element type — 2 bf16, 3 e5m2 (the codes widened to FP32 with the K/V
// scales applied; the query unquantised and P exact, as on bf16 layers).
template <int D, int ELT, int G>
struct DecodeCfg {
  static_assert(ELT == 2 || ELT == 3, "bf16 or e5m2 pools");
  static constexpr int ES = ELT == 2 ? 2 : 1;                 // bytes per element
  static constexpr int CHUNK = 16 * D * ES;                   // bytes of one (block, head) chunk
  static constexpr int TB = CHUNK <= 2048 ? 2 : 1;            // 16-key blocks per tile
  static constexpr int TILE_BYTES = TB * 2 * CHUNK;           // K and V of a tile
  static constexpr int RING = kNW * kNBUF * TILE_BYTES;
  // QK mapping: EPL elements (EPL*ES bytes) of one key per lane
  static constexpr int EPL = G <= 8 ? 8 : 4;
  static constexpr int LPK = D / EPL;                         // lanes per key
  static constexpr int KPR = 32 / LPK;                        // keys per round
  static constexpr int ROUNDS = 16 / KPR;                     // rounds per block
  static constexpr int NVF = G > LPK ? G / LPK : 1;           // scores per lane per round
  // PV mapping: VPL elements of one value row per lane
  static constexpr int VPL0 = G <= 4 ? 4 : 2;
  static constexpr int VPL = VPL0 > D / 32 ? VPL0 : D / 32;
  static constexpr int LPV = D / VPL;                         // lanes per value row
  static constexpr int KPV = 32 / LPV;                        // keys in parallel
  static constexpr int MIN_CTAS = (G * D <= 512 && RING <= 65536) ? 3 : 2;
  static_assert(LPK >= 2 && LPK <= 32, "lanes per key");
  static_assert(LPV >= 1 && LPV <= 32, "lanes per value row");
  static_assert(G * VPL <= 64 && G * EPL <= 64, "register budget");
  static_assert(NVF == 1, "every lane ends the QK reduction with one whole score");
  static_assert(kNW * G * D * 4 <= RING, "the warps' accumulators are merged inside the ring");
  static_assert(RING / 4 >= 2 * G + 8 * G, "the merge keeps at least 8 split weights per head in the ring");
};

template <int N>
FKV_DEV void load_bytes(const uint8_t* p, uint32_t (&w)[N / 4 > 0 ? N / 4 : 1]) {
  if constexpr (N == 16) {
    const uint4 x = *reinterpret_cast<const uint4*>(p);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
  } else if constexpr (N == 8) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    w[0] = x.x; w[1] = x.y;
  } else if constexpr (N == 4) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else {
    w[0] = *reinterpret_cast<const uint16_t*>(p);
  }
}

// Convert N elements (bf16 or e5m2) held in words to float2 pairs.
template <int ELT, int N>
FKV_DEV void to_f2(const uint32_t* w, float2* out) {
  if constexpr (ELT == 3) {
    if constexpr (N >= 4) {
#pragma unroll
      for (int i = 0; i < N / 4; ++i) e5m2x4_to_f2(w[i], out[2 * i], out[2 * i + 1]);
    } else {
      float2 unused;
      e5m2x4_to_f2(w[0] & 0xFFFFu, out[0], unused);
    }
  } else {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) out[i] = bf16x2_to_f2(w[i]);
  }
}

// fp8_decode_step on a bf16 (skip) or e5m2 layer: the current token's K and V rows of KV
// head g written into the pools at position T - 1 exactly as kv_quant_cache writes them
// (bf16: a copy; e5m2: e5m2(fl32(x * fl32(1 / s))), round to nearest even, saturating).
// Threads j < 2 D / 8 of the CTA take 8 elements of K (j < D / 8) or V each; each writer
// fences its stores against the async proxy, and the CTA barrier that follows orders
// them before the bulk copies that read the block back.
template <int D, int ELT>
__device__ void write_current_token_cc(const DecodeParams& p, int b, int g, int T) {
  const int pos = T - 1;
  const int id = p.block_table[static_cast<size_t>(b) * p.max_blocks + (pos >> 4)];
  if (id < 0 || id >= p.num_blocks) return;  // reported by the block-id checks of the split
  constexpr int CH = D / 8;
  const int j = threadIdx.x;
  if (j >= 2 * CH) return;
  const bool is_v = j >= CH;
  const int c = is_v ? j - CH : j;
  const size_t elem = ((static_cast<size_t>(id) * p.Hkv + g) * 16 + (pos & 15)) * D + 8 * c;
  const uint4 x = reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) + (static_cast<size_t>(b) * p.Hkv + g) * D)[c];
  // the pools are the caller's writable device memory; the params carry them as const
  // because the plain decode only reads them
  uint8_t* pool = const_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache);
  if constexpr (ELT == 2) {
    *reinterpret_cast<uint4*>(pool + 2 * elem) = x;
  } else {
    const float inv = __frcp_rn((is_v ? p.v_scale : p.k_scale)[p.per_head ? g : 0]);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 f0 = bf16x2_to_f2(w[2 * k]), f1 = bf16x2_to_f2(w[2 * k + 1]);
      o[k] = static_cast<uint32_t>(f32x2_to_e5m2x2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv))) |
             (static_cast<uint32_t>(f32x2_to_e5m2x2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv))) << 16);
    }
    *reinterpret_cast<uint2*>(pool + elem) = make_uint2(o[0], o[1]);
  }
  fence_proxy_async_global();
}

template <int D, int ELT, int G>
__global__ void __launch_bounds__(kNW * 32, DecodeCfg<D, ELT, G>::MIN_CTAS)
    decode_split_kernel(const DecodeParams p) {
  using C = DecodeCfg<D, ELT, G>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING);             // [NW][NBUF]
  float* p_s = reinterpret_cast<float*>(full + kNW * kNBUF);                // [NW][16*TB][G]
  float* alpha_s = p_s + kNW * 16 * C::TB * G;                              // [NW][G]
  float* ml_s = alpha_s + kNW * G;                                          // [NW][2][G]
  int* ids_s = reinterpret_cast<int*>(ml_s + kNW * 2 * G);                  // [kMaxBps]

  const int sigma = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next kernel in the stream may be scheduled as this grid's CTAs finish; the
  // barriers need no input and are set up before waiting for the kernels before this one
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNW * kNBUF; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  griddep_wait();
  const SeqRange r = seq_range(p, b, sigma == 0 && g == 0 && threadIdx.x == 0);
  if (sigma >= r.nsplit) {  // uniform over the CTA
    if (sigma == 0) {  // a sequence without keys: zero output rows
      for (int t = threadIdx.x; t < G * D; t += blockDim.x)
        p.out[(static_cast<size_t>(b) * p.Hq + g * G + t / D) * D + t % D] = __float2bfloat16(0.f);
    }
    return;
  }
  const int blk_first = r.blk_begin + sigma * p.bps;
  const int nblk = min(p.bps, r.blk_end - blk_first);
  const int ntiles = (nblk + C::TB - 1) / C::TB;

  {
    const int* row = p.block_table + static_cast<size_t>(b) * p.max_blocks + blk_first;
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
      int id = row[i];
      if (id < 0 || id >= p.num_blocks) {
        raise_fault(p.fault, FKV_FAULT_BLOCK_ID);
        id = 0;
      }
      ids_s[i] = id;
    }
  }
  // fp8_decode_step: the split holding position T - 1 (the last) writes the current token
  // into the pools before any copy of that block is issued (not when the context was clamped)
  if (p.k_new != nullptr && sigma == r.nsplit - 1 && !r.clamped) write_current_token_cc<D, ELT>(p, b, g, r.T);
  __syncthreads();

  // ---------------------------------------------------------------- per-warp pipeline
  uint64_t* wfull = full + warp * kNBUF;
  uint8_t* wring = ring + warp * kNBUF * C::TILE_BYTES;
  // the k-th tile of this warp is tile warp + k*NW, in buffer k % NBUF
  auto issue = [&](int k) {
    const int t = warp + k * kNW;
    if (t >= ntiles) return;
    const int b0 = t * C::TB;
    const int nb = min(C::TB, nblk - b0);
    uint64_t* bar = &wfull[k % kNBUF];
    uint8_t* dst = wring + (k % kNBUF) * C::TILE_BYTES;
    mbar_arrive_expect_tx(bar, nb * 2 * C::CHUNK);
    for (int j = 0; j < nb; ++j) {
      const size_t off = (static_cast<size_t>(ids_s[b0 + j]) * p.Hkv + g) * C::CHUNK;
      bulk_g2s(dst + j * 2 * C::CHUNK, p.k_cache + off, C::CHUNK, bar);
      bulk_g2s(dst + j * 2 * C::CHUNK + C::CHUNK, p.v_cache + off, C::CHUNK, bar);
    }
  };
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kNBUF; ++k) issue(k);
  }

  const int h0 = g * G;
  const int kq = lane / C::LPK;                 // key within a QK round
  const int dq = (lane % C::LPK) * C::EPL;      // first element of the lane's QK slice
  const int vg = lane / C::LPV;                 // key sub-group of the PV mapping
  const int dv = (lane % C::LPV) * C::VPL;      // first element of the lane's PV slice

  // Heads of a lane.  The transposing reduction below halves the lane's G partial dot
  // products at every shuffle level, keeping the lower half of its slots and receiving
  // the partner's upper half.  For that to need no selects, lane slot j holds query head
  // j ^ hb, where hb collects the lane bits of the halving levels; after the reduction
  // slot 0 holds the full score of head hb.
  int hb = 0;
  {
    int nv = G;
#pragma unroll
    for (int off = C::LPK / 2; off >= 1; off >>= 1) {
      if (nv > 1) {
        if (lane & off) hb += nv / 2;
        nv >>= 1;
      }
    }
  }
  const bool dup0 = (C::LPK <= G) ? true : ((lane % C::LPK) % (C::LPK / G) == 0);
  // softmax constant: softmax_scale * log2(e), times the K scale on e5m2 layers
  const float cl = p.sm_scale_log2 * (ELT == 3 ? p.k_scale[p.per_head ? g : 0] : 1.f);
  // query slice in slot order, FP32
  float2 qf[G][C::EPL / 2];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int h = j ^ hb;
    const __nv_bfloat16* qp = p.q + (static_cast<size_t>(b) * p.Hq + h0 + h) * D + dq;
#pragma unroll
    for (int e = 0; e < C::EPL / 2; ++e) qf[j][e] = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(qp + 2 * e));
  }

  float m_run = -INFINITY, l_run = 0.f;
  float2 acc[G][C::VPL / 2 > 0 ? C::VPL / 2 : 1];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < C::VPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);

  // per-warp probabilities of the current tile, one float per (key, head)
  float* pw = p_s + warp * 16 * C::TB * G;
  float* aw = alpha_s + warp * G;
  int issued = min(kNBUF, max(0, (ntiles - warp + kNW - 1) / kNW));
  int k = 0;
  bool timed_out = false;
  for (;; ++k) {
    const int t = warp + k * kNW;
    if (t >= ntiles) break;
    const int buf = k % kNBUF;
    if (!mbar_wait_bounded(&wfull[buf], (k / kNBUF) & 1)) {
      raise_fault(p.fault, FKV_FAULT_TIMEOUT);
      timed_out = true;
      break;
    }
    const uint8_t* tile = wring + buf * C::TILE_BYTES;
    const int nb = min(C::TB, nblk - t * C::TB);
    const int key0 = (blk_first + t * C::TB) * 16;  // absolute position of the tile's first key
    const bool interior = nb == C::TB && key0 >= r.lo && key0 + 16 * C::TB <= r.T;

    // ---------------- QK
    float sc[C::TB][C::ROUNDS];
    auto qk = [&](auto all_valid) {
#pragma unroll
      for (int j = 0; j < C::TB; ++j) {
        const uint8_t* kb = tile + j * 2 * C::CHUNK;
#pragma unroll
        for (int rr = 0; rr < C::ROUNDS; ++rr) {
          const int key = rr * C::KPR + kq;
          uint32_t w[C::EPL * C::ES / 4 > 0 ? C::EPL * C::ES / 4 : 1];
          load_bytes<C::EPL * C::ES>(kb + key * D * C::ES + dq * C::ES, w);
          float v[G];
          float2 kf[C::EPL / 2];
          to_f2<ELT, C::EPL>(w, kf);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < C::EPL / 2; ++e) a = __ffma2_rn(qf[h][e], kf[e], a);
            v[h] = a.x + a.y;
          }
          // select-free transposing reduction across the LPK lanes of this key
          int nv = G;
#pragma unroll
          for (int off = C::LPK / 2; off >= 1; off >>= 1) {
            if (nv > 1) {
#pragma unroll
              for (int q2 = 0; q2 < nv / 2; ++q2) v[q2] += __shfl_xor_sync(0xffffffffu, v[q2 + nv / 2], off);
              nv >>= 1;
            } else {
              v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
            }
          }
          if constexpr (decltype(all_valid)::value) {
            sc[j][rr] = v[0] * cl;
          } else {
            const int kabs = key0 + j * 16 + key;
            const bool valid = j < nb && kabs >= r.lo && kabs < r.T;
            sc[j][rr] = valid ? v[0] * cl : -INFINITY;
          }
        }
      }
    };
    if (interior) qk(std::true_type{});
    else qk(std::false_type{});

    // ---------------- softmax (base 2) over the tile's keys
    {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < C::TB; ++j)
#pragma unroll
        for (int rr = 0; rr < C::ROUNDS; ++rr) mx = fmaxf(mx, sc[j][rr]);
#pragma unroll
      for (int off = C::LPK; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m_run, mx);
      const float alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - mn);
      m_run = mn;
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < C::TB; ++j)
#pragma unroll
        for (int rr = 0; rr < C::ROUNDS; ++rr) {
          const float pv = ex2(sc[j][rr] - mn);
          sum += pv;
          if (dup0) pw[(j * 16 + rr * C::KPR + kq) * G + hb] = pv;
        }
#pragma unroll
      for (int off = C::LPK; off < 32; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run = l_run * alpha + sum;
      if (dup0 && kq == 0) aw[hb] = alpha;
    }
    __syncwarp();

    // ---------------- PV
    {
      bool rescale = false;
#pragma unroll
      for (int h = 0; h < G; ++h) rescale |= (aw[h] != 1.f);
      if (rescale) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float2 a2 = make_float2(aw[h], aw[h]);
#pragma unroll
          for (int e = 0; e < C::VPL / 2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], a2);
        }
      }
    }
    // P.V in FP32
#pragma unroll
    for (int j = 0; j < C::TB; ++j) {
      if (j >= nb) break;
      const uint8_t* vb = tile + j * 2 * C::CHUNK + C::CHUNK;
      // keys of this block inside [lo, T); the bytes of the other keys may be stale (even
      // NaN codes), so they are skipped rather than weighted by p = 0.
      const int kb0 = key0 + j * 16;
      const int kv_lo = max(r.lo - kb0, 0), kv_hi = min(r.T - kb0, 16);
      auto pv_key = [&](int key) {
        uint32_t w[C::VPL * C::ES / 4 > 0 ? C::VPL * C::ES / 4 : 1];
        load_bytes<C::VPL * C::ES>(vb + key * D * C::ES + dv * C::ES, w);
        const int pidx = (j * 16 + key) * G;
        float2 vf[C::VPL / 2];
        to_f2<ELT, C::VPL>(w, vf);
        float pv[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int h = 0; h < G; h += 4) {
            const float4 x = *reinterpret_cast<const float4*>(pw + pidx + h);
            pv[h] = x.x; pv[h + 1] = x.y; pv[h + 2] = x.z; pv[h + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) pv[h] = pw[pidx + h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float2 p2 = make_float2(pv[h], pv[h]);
#pragma unroll
          for (int e = 0; e < C::VPL / 2; ++e) acc[h][e] = __ffma2_rn(p2, vf[e], acc[h][e]);
        }
      };
      if (kv_lo == 0 && kv_hi == 16) {
#pragma unroll
        for (int kk = 0; kk < 16 / C::KPV; ++kk) pv_key(kk * C::KPV + vg);
      } else {
#pragma unroll
        for (int kk = 0; kk < 16 / C::KPV; ++kk) {
          const int key = kk * C::KPV + vg;
          if (key >= kv_lo && key < kv_hi) pv_key(key);
        }
      }
    }
    __syncwarp();
    // the buffer is free again: refill it with this warp's tile k + NBUF
    if (lane == 0) {
      fence_proxy_async_smem();
      issue(k + kNBUF);
    }
    if (warp + (k + kNBUF) * kNW < ntiles) ++issued;
  }
  if (timed_out && lane == 0) {
    // let the copies still in flight land before the CTA can exit
    for (int kk = k; kk < issued; ++kk) mbar_wait_bounded(&wfull[kk % kNBUF], (kk / kNBUF) & 1);
  }

  // reduce the key sub-groups of the PV mapping
#pragma unroll
  for (int off = C::LPV; off < 32; off <<= 1) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < C::VPL / 2; ++e) {
        acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, off);
        acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, off);
      }
  }
  if (dup0 && kq == 0) {
    ml_s[(warp * 2 + 0) * G + hb] = m_run;
    ml_s[(warp * 2 + 1) * G + hb] = l_run;
  }
  __syncthreads();  // every warp is done with the ring and has no copy in flight
  float* acc_w = reinterpret_cast<float*>(ring);  // [NW][G][D]
  if (vg == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < C::VPL / 2; ++e)
        *reinterpret_cast<float2*>(acc_w + (warp * G + h) * D + dv + 2 * e) = acc[h][e];
  }
  __syncthreads();

  // ---------------------------------------------------- merge the warps, write the split
  for (int t = threadIdx.x; t < G * D; t += blockDim.x) {
    const int h = t / D, d = t % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kNW; ++w) M = fmaxf(M, ml_s[(w * 2) * G + h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kNW; ++w) {
        const float mw = ml_s[(w * 2) * G + h];
        if (mw == -INFINITY) continue;
        const float fw = ex2(mw - M);
        L += ml_s[(w * 2 + 1) * G + h] * fw;
        O += acc_w[(w * G + h) * D + d] * fw;
      }
    }
    const size_t row = (static_cast<size_t>(b) * p.Hq + g * G + h) * p.max_splits + sigma;
    p.o_part[row * D + d] = L > 0.f ? O / L : 0.f;
    if (d == 0) p.lse_part[row] = L > 0.f ? M + lg2(L) : -INFINITY;
  }

  // ---------------------------------------------------- the last split of (b, g) merges
  // o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M), times the V scale, to bf16: the
  // FP32 second level of the accumulation.
  volatile int* last_s = ids_s;  // the block ids are no longer needed
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *last_s = count_split_done(p, b * p.Hkv + g, r.nsplit);
  __syncthreads();
  if (!*last_s) return;
  __threadfence();
  constexpr int CH = (C::RING / 4 - 2 * G) / G < 256 ? (C::RING / 4 - 2 * G) / G : 256;
  merge_splits<D, G, kNW * 32, CH>(p, b, g, r.nsplit, ELT == 3 ? p.v_scale[p.per_head ? g : 0] : 1.f,
                                   reinterpret_cast<float*>(ring));
}

template <int D, int ELT, int G>
size_t decode_smem_bytes() {
  using C = DecodeCfg<D, ELT, G>;
  return C::RING + kNW * kNBUF * sizeof(uint64_t) +
         (kNW * 16 * C::TB * G + kNW * G + kNW * 2 * G) * sizeof(float) + kMaxBps * sizeof(int);
}

template <int D, int ELT, int G>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  const size_t smem = decode_smem_bytes<D, ELT, G>();
  auto kern = decode_split_kernel<D, ELT, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_splits, p.Hkv, p.B);
  return launch_dependent(kern, grid, dim3(kNW * 32), smem, s, p);
}

template <int D, int ELT>
cudaError_t launch_decode_g(const DecodeParams& p, int G, cudaStream_t s) {
  switch (G) {
    case 1: return launch_decode_t<D, ELT, 1>(p, s);
    case 2: return launch_decode_t<D, ELT, 2>(p, s);
    case 4: return launch_decode_t<D, ELT, 4>(p, s);
    case 8: return launch_decode_t<D, ELT, 8>(p, s);
    case 16:
      if constexpr (D <= 128) return launch_decode_t<D, ELT, 16>(p, s);
      else return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, int elt, int G, cudaStream_t s) {
  if (elt == 2) return launch_decode_g<D, 2>(p, G, s);
  if (elt == 3) return launch_decode_g<D, 3>(p, G, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams& p, int D, int elt, int G, cudaStream_t s) {
  if (D == 64) return launch_decode_d<64>(p, elt, G, s);
  if (D == 128) return launch_decode_d<128>(p, elt, G, s);
  if (D == 256) return launch_decode_d<256>(p, elt, G, s);
  return cudaErrorInvalidValue;
}

}  // namespace fkv
