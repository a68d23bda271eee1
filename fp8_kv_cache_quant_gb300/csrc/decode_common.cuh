// Pieces shared by the split-K decode kernels: the per-sequence key range in pool blocks
// and the FP32 merge of the splits' partial results.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace fkv {

// Keys [lo, T) of sequence b, as blocks [blk_begin, blk_end), in nsplit splits of p.bps
// blocks.  A context longer than the block table can address is clamped (and reported).
// `clamped` marks a context length outside [0, max_blocks * 16]: the fused cache write of
// fp8_decode_step then writes nothing (position T - 1 of the clamped range is a cached
// token of the caller's, not the current one).
struct SeqRange {
  int T, lo, blk_begin, blk_end, nsplit;
  bool clamped;
};

FKV_DEV SeqRange seq_range(const DecodeParams& p, int b, bool report) {
  SeqRange r;
  int T = p.context_lens[b];
  const int cap = p.max_blocks * 16;
  r.clamped = T < 0 || T > cap;
  if (r.clamped) {
    if (report) raise_fault(p.fault, FKV_FAULT_CONTEXT);
    T = T < 0 ? 0 : cap;
  }
  r.T = T;
  r.lo = p.window > 0 ? max(0, T - p.window) : 0;
  r.blk_begin = r.lo >> 4;
  r.blk_end = (T + 15) >> 4;
  const int nb = r.blk_end - r.blk_begin;
  r.nsplit = nb > 0 ? (nb + p.bps - 1) / p.bps : 0;
  return r;
}

// One split of unit u (a sequence's KV head) is done: count it.  Returns true for the
// split that completes the unit, whose CTA then merges; that CTA also returns the counter
// to zero, since every other split has counted, so the workspace's counters are zero
// again for the next call.  A count already at nsplit or beyond means the counters were
// not zero when the call began (a workspace not zero-filled before first use).
FKV_DEV bool count_split_done(const DecodeParams& p, int u, int nsplit) {
  const int old = atomicAdd(&p.done[u], 1);
  if (old >= nsplit) raise_fault(p.fault, FKV_FAULT_WORKSPACE);
  if (old != nsplit - 1) return false;
  p.done[u] = 0;
  return true;
}

// The second, FP32 level of the split-K accumulation, run by the CTA that finished the
// last split of (sequence b, KV head g): with lse_s the base-2 log-sum-exp of split s
// and o_s its normalised output, o = v_s * sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),
// M = max_s lse_s, written as bf16.  Every thread of the CTA calls it (it synchronises);
// `scratch` holds at least 2 * G + G * CH floats of shared memory.
// The partials come from L2; a load whose value the next instruction needs holds the
// warp for the whole round trip.  With at most eight splits and one group of four
// outputs per thread, each thread issues all its loads (its head's log-sum-exps and its
// outputs' partials) at once and merges alone: one round trip.  Otherwise the
// log-sum-exps are read by a warp per head with the lanes striding over the splits, and
// each group of four outputs' split partials are loaded sixteen at a time (16-byte
// loads) before they are summed.  Both sum the outputs in split order and the weights
// in the same pairwise order, so they give the same bits.
template <int D, int G, int NT, int CH>
FKV_DEV void merge_splits(const DecodeParams& p, int b, int g, int ns, float vs, float* scratch) {
  constexpr int QUADS = (G * D / 4 + NT - 1) / NT;  // groups of 4 outputs per thread
  constexpr int UF = 8;  // splits merged in one round trip (every load issued at once)
  static_assert(UF == 8, "the pairwise weight sum below is written for eight splits");
  if (ns <= UF && QUADS == 1) {
    // few splits: each thread loads its four outputs of every split and its head's
    // log-sum-exps together, then merges them itself
    const int t = threadIdx.x;
    if (t < G * D / 4) {
      const int h = t / (D / 4), d = 4 * (t % (D / 4));
      const size_t row = (static_cast<size_t>(b) * p.Hq + g * G + h) * p.max_splits;
      const float* src = p.o_part + row * D + d;
      float4 x[UF];
      float lv[UF];
#pragma unroll
      for (int u = 0; u < UF; ++u) {
        if (u < ns) {
          x[u] = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(u) * D));
          lv[u] = __ldcg(p.lse_part + row + u);
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int u = 0; u < UF; ++u)
        if (u < ns) M = fmaxf(M, lv[u]);
      float w[UF];
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < UF; ++u) w[u] = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int u = 0; u < UF; ++u) {
          if (u < ns) {
            const float wv = (lv[u] == -INFINITY) ? 0.f : ex2(lv[u] - M);
            w[u] = wv;
            o.x += wv * x[u].x;
            o.y += wv * x[u].y;
            o.z += wv * x[u].z;
            o.w += wv * x[u].w;
          }
        }
      }
      // the weights summed pairwise in the order of a warp's butterfly over eight lanes,
      // as the general path below sums them
      const float W = ((w[0] + w[4]) + (w[2] + w[6])) + ((w[1] + w[5]) + (w[3] + w[7]));
      const float inv = (W > 0.f) ? vs / W : 0.f;
      __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(p.out + (static_cast<size_t>(b) * p.Hq + g * G + h) * D + d);
      dst[0] = __floats2bfloat162_rn(o.x * inv, o.y * inv);
      dst[1] = __floats2bfloat162_rn(o.z * inv, o.w * inv);
    }
    return;
  }
  float* ms_s = scratch;       // [G] max of lse
  float* inv_s = ms_s + G;     // [G] v_s / sum of weights
  float* w_s = inv_s + G;      // [G][CH] weights of a chunk of splits
  constexpr int NWARP = NT / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row_base = (static_cast<size_t>(b) * p.Hq + g * G) * p.max_splits;
  for (int h = warp; h < G; h += NWARP) {
    const float* lse = p.lse_part + row_base + static_cast<size_t>(h) * p.max_splits;
    float M = -INFINITY;
    for (int s2 = lane; s2 < ns; s2 += 32) M = fmaxf(M, __ldcg(lse + s2));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float W = 0.f;
    if (M != -INFINITY)
      for (int s2 = lane; s2 < ns; s2 += 32) {
        const float lv = __ldcg(lse + s2);
        W += (lv == -INFINITY) ? 0.f : ex2(lv - M);
      }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    if (lane == 0) {
      ms_s[h] = M;
      inv_s[h] = (W > 0.f) ? vs / W : 0.f;
    }
  }
  constexpr int U = 16;                              // split partials loaded before use
  float4 o[QUADS];
#pragma unroll
  for (int k2 = 0; k2 < QUADS; ++k2) o[k2] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < ns; c0 += CH) {
    const int nc = min(CH, ns - c0);
    __syncthreads();
    for (int t = threadIdx.x; t < G * nc; t += NT) {
      const int h = t / nc, j = t % nc;
      const float lv = __ldcg(p.lse_part + row_base + static_cast<size_t>(h) * p.max_splits + c0 + j);
      w_s[h * CH + j] = (lv == -INFINITY) ? 0.f : ex2(lv - ms_s[h]);
    }
    __syncthreads();
#pragma unroll
    for (int k2 = 0; k2 < QUADS; ++k2) {
      const int t = threadIdx.x + k2 * NT;
      if (t < G * D / 4) {
        const int h = t / (D / 4), d = 4 * (t % (D / 4));
        const float* src = p.o_part + (row_base + static_cast<size_t>(h) * p.max_splits + c0) * D + d;
        const float* wh = w_s + h * CH;
        int j = 0;
        for (; j + U <= nc; j += U) {
          float4 x[U];
#pragma unroll
          for (int u = 0; u < U; ++u) x[u] = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(j + u) * D));
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const float wv = wh[j + u];
            o[k2].x += wv * x[u].x;
            o[k2].y += wv * x[u].y;
            o[k2].z += wv * x[u].z;
            o[k2].w += wv * x[u].w;
          }
        }
        for (; j < nc; ++j) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(j) * D));
          const float wv = wh[j];
          o[k2].x += wv * x.x;
          o[k2].y += wv * x.y;
          o[k2].z += wv * x.z;
          o[k2].w += wv * x.w;
        }
      }
    }
  }
#pragma unroll
  for (int k2 = 0; k2 < QUADS; ++k2) {
    const int t = threadIdx.x + k2 * NT;
    if (t < G * D / 4) {
      const int h = t / (D / 4), d = 4 * (t % (D / 4));
      const float inv = inv_s[h];
      __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(p.out + (static_cast<size_t>(b) * p.Hq + g * G + h) * D + d);
      dst[0] = __floats2bfloat162_rn(o[k2].x * inv, o[k2].y * inv);
      dst[1] = __floats2bfloat162_rn(o[k2].z * inv, o[k2].w * inv);
    }
  }
}

}  // namespace fkv
