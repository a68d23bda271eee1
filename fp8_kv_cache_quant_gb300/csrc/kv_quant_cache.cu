// kv_quant_cache: bf16 K/V of new tokens -> paged e4m3 (or e5m2) pool, or a bf16 copy for
// skip layers.  The cache write of the vLLM blog "FP8 KV-Cache and Attention quantization
// in vLLM" (section "Kernel 与 vLLM 改进", paragraph "Per-Head Scales": the write takes a
// per-KV-head scale array instead of one scalar; paragraph "跳过 Layer": skipped layers
// stay bf16).
//
// One thread handles 8 consecutive elements of one (token, head) row of K and of V:
// a 16-byte load of each, 8-byte e4m3 stores (16-byte for bf16).  Consecutive threads
// cover consecutive 16-byte pieces, so loads and stores coalesce.  HBM-bound.
// The counting instantiation also counts the elements whose scaled value lies beyond
// +-448 and is clipped by the saturating encode (the clipping frequency the KV-cache
// quantisation explainer asks to watch): per thread, then one atomic add per warp.
#include "common.cuh"
#include "kernels.h"

namespace fkv {

template <bool kBf16, bool kCount, bool kE5>
__global__ void __launch_bounds__(256) kv_quant_cache_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    int n_tokens, int H, int D, uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
    long long capacity, const float* __restrict__ ks, const float* __restrict__ vs, int per_head,
    int32_t* fault, unsigned long long* clips) {
  const int chunks = D >> 3;
  unsigned int kclip = 0, vclip = 0;
  const long long total = static_cast<long long>(n_tokens) * H * chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % chunks);
    const long long th = i / chunks;
    const int h = static_cast<int>(th % H);
    const long long t = th / H;
    const long long slot = slots[t];
    if (slot < 0) continue;
    if (slot >= capacity) {
      if (h == 0 && c == 0) raise_fault(fault, FKV_FAULT_SLOT);
      continue;
    }
    const long long blk = slot >> 4, off = slot & 15;
    const long long dst = (((blk * H + h) << 4) + off) * D + (c << 3);  // element index
    const uint4 kx = k[i];
    const uint4 vx = v[i];
    if constexpr (kBf16) {
      reinterpret_cast<uint4*>(kc)[dst >> 3] = kx;
      reinterpret_cast<uint4*>(vc)[dst >> 3] = vx;
    } else {
      const float ik = __frcp_rn(ks[per_head ? h : 0]);
      const float iv = __frcp_rn(vs[per_head ? h : 0]);
      const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
      const uint32_t vw[4] = {vx.x, vx.y, vx.z, vx.w};
      uint32_t ko[2], vo[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 k0 = bf16x2_to_f2(kw[2 * j]), k1 = bf16x2_to_f2(kw[2 * j + 1]);
        const float2 v0 = bf16x2_to_f2(vw[2 * j]), v1 = bf16x2_to_f2(vw[2 * j + 1]);
        const float ky[4] = {__fmul_rn(k0.x, ik), __fmul_rn(k0.y, ik), __fmul_rn(k1.x, ik), __fmul_rn(k1.y, ik)};
        const float vy[4] = {__fmul_rn(v0.x, iv), __fmul_rn(v0.y, iv), __fmul_rn(v1.x, iv), __fmul_rn(v1.y, iv)};
        constexpr float kLimit = kE5 ? 57344.f : 448.f;  // largest finite code of the format
        if constexpr (kCount) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            kclip += fabsf(ky[e]) > kLimit ? 1u : 0u;  // NaN compares false: not a clip
            vclip += fabsf(vy[e]) > kLimit ? 1u : 0u;
          }
        }
        auto enc = [](float a, float b2) -> uint32_t {
          if constexpr (kE5) return f32x2_to_e5m2x2(a, b2);
          else return f32x2_to_e4m3x2(a, b2);
        };
        const uint32_t klo = enc(ky[0], ky[1]);
        const uint32_t khi = enc(ky[2], ky[3]);
        const uint32_t vlo = enc(vy[0], vy[1]);
        const uint32_t vhi = enc(vy[2], vy[3]);
        ko[j] = klo | (khi << 16);
        vo[j] = vlo | (vhi << 16);
      }
      reinterpret_cast<uint2*>(kc)[dst >> 3] = make_uint2(ko[0], ko[1]);
      reinterpret_cast<uint2*>(vc)[dst >> 3] = make_uint2(vo[0], vo[1]);
    }
  }
  if constexpr (kCount) {
    // every lane of the warp reaches this point (no early return above)
    kclip = __reduce_add_sync(0xffffffffu, kclip);
    vclip = __reduce_add_sync(0xffffffffu, vclip);
    if ((threadIdx.x & 31) == 0 && (kclip | vclip) != 0) {
      atomicAdd(clips, static_cast<unsigned long long>(kclip));
      atomicAdd(clips + 1, static_cast<unsigned long long>(vclip));
    }
  }
}

cudaError_t launch_kv_quant_cache(const void* k, const void* v, const int64_t* slots, int n_tokens,
                                  const fkv_layer_cache& cache, const float* ks, const float* vs,
                                  int per_head, bool bf16_layer, int32_t* fault, cudaStream_t s,
                                  int num_sms, unsigned long long* clips) {
  const bool e5 = !bf16_layer && cache.kv_format == FKV_KV_E5M2;
  const long long total = static_cast<long long>(n_tokens) * cache.num_kv_heads * (cache.head_dim / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const long long capacity = static_cast<long long>(cache.num_blocks) * cache.block_size;
  auto kern = bf16_layer ? kv_quant_cache_kernel<true, false, false>
               : e5      ? (clips != nullptr ? kv_quant_cache_kernel<false, true, true>
                                             : kv_quant_cache_kernel<false, false, true>)
                         : (clips != nullptr ? kv_quant_cache_kernel<false, true, false>
                                             : kv_quant_cache_kernel<false, false, false>);
  kern<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, n_tokens, cache.num_kv_heads, cache.head_dim,
      static_cast<uint8_t*>(cache.k_cache), static_cast<uint8_t*>(cache.v_cache), capacity, ks, vs, per_head, fault,
      clips);
  return cudaGetLastError();
}

}  // namespace fkv
