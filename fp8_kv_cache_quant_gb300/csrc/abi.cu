// The C ABI of libfp8kv.so: argument validation, launch planning and dispatch.
// Nothing here allocates memory or keeps state between calls.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace {

using fkv::DecodeParams;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int current_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // no device: plan for a full GB300
    n = 152;
  }
  return n;
}

bool layer_is_bf16(int32_t layer, const uint8_t* mask, int32_t num_layers, fkv_status* st) {
  if (mask == nullptr) return false;
  if (layer < 0 || layer >= num_layers) {
    *st = FKV_INVALID_ARG;
    return false;
  }
  return mask[layer] != 0;
}

bool supported_head_dim(int32_t d) { return d == 64 || d == 128 || d == 256; }

bool valid_format(const fkv_layer_cache& c) { return c.kv_format == FKV_KV_E4M3 || c.kv_format == FKV_KV_E5M2; }

// Element type of a layer's pools for the decode kernels: 1 e4m3, 2 bf16, 3 e5m2.
int layer_elt(bool bf16, const fkv_layer_cache& c) { return bf16 ? 2 : (c.kv_format == FKV_KV_E5M2 ? 3 : 1); }

bool supported_group(int32_t G, int32_t D) {
  if (!(G == 1 || G == 2 || G == 4 || G == 8 || G == 16)) return false;
  return G * D <= 2048;
}

// Pool blocks per tile of the tensor-core decode (its P-rounding granularity): 128 keys,
// 256 at head_dim 64.  The split plan keeps whole tiles for every layer kind.
int decode_tile_blocks(int32_t D) { return D == 64 ? 16 : 8; }

struct DecodePlan {
  int bps = 0;
  int max_splits = 0;
  size_t o_bytes = 0, lse_bytes = 0, cnt_bytes = 0;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Split-K plan.  Blocks per split (bps) are multiples of the tensor-core decode's tile (8
// blocks of 16 keys; 16 at head_dim 64) up to kMaxSplitBlocks (256), with at most 1024
// splits per sequence.
// Equal estimates go to the longer splits (fewer CTAs, fewer prologues and merges).  A requested
// num_splits sets bps = ceil(blocks / num_splits), rounded up.  Otherwise bps minimises
// the estimated time waves * bps, where a wave is one CTA on every resident slot
// (3 per SM) and the grid has B * Hkv * ceil(blocks / bps) CTAs: the longest split
// sets a wave's time, and a partly filled last wave costs as much as a full one.
bool plan_decode(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t max_blocks, int32_t window,
                 int32_t num_splits, DecodePlan* plan) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_blocks <= 0 || window < 0 || num_splits < 0) return false;
  long long nblk_max = max_blocks;
  if (window > 0) nblk_max = std::min<long long>(max_blocks, (window + 15) / 16 + 1);
  const long long tpb = decode_tile_blocks(D);
  long long bps;
  if (num_splits > 0) {
    bps = (nblk_max + num_splits - 1) / num_splits;
  } else {
    const long long units = static_cast<long long>(std::max(B, 1)) * Hkv;
    const long long slots = static_cast<long long>(current_num_sms()) * 3;
    long long best = -1, best_cost = 0;
    for (long long c = tpb; c <= fkv::kMaxSplitBlocks; c += tpb) {
      const long long ctas = units * ((nblk_max + c - 1) / c);
      const long long cost = (ctas + slots - 1) / slots * std::min(c, nblk_max);
      if (best < 0 || cost < best_cost || (cost == best_cost && c > best)) {
        best = c;
        best_cost = cost;
      }
    }
    bps = best;
  }
  bps = std::min<long long>(bps, fkv::kMaxSplitBlocks);
  bps = std::max<long long>(bps, (nblk_max + 1023) / 1024);
  bps = std::max<long long>(bps, 1);
  bps = (bps + tpb - 1) / tpb * tpb;
  if (bps > fkv::kMaxSplitBlocks) return false;  // context too long for 1024 splits of 256 blocks
  plan->bps = static_cast<int>(bps);
  plan->max_splits = static_cast<int>((nblk_max + bps - 1) / bps);
  const size_t rows = static_cast<size_t>(B) * Hq * plan->max_splits;
  plan->o_bytes = align256(rows * D * sizeof(float));
  plan->lse_bytes = align256(rows * sizeof(float));
  plan->cnt_bytes = align256(static_cast<size_t>(std::max(B, 1)) * Hkv * sizeof(int32_t));
  return true;
}

fkv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FKV_OK : FKV_CUDA_ERROR; }

// Bound of the tensor-core decode's pipeline waits set by fkv_set_decode_wait_limit_ns;
// 0 = the default (kPipeWaitNs).
std::atomic<unsigned long long> g_decode_wait_ns{0};
constexpr unsigned long long kDefaultPipeWaitNs = 200000000ull;  // 200 ms, as kPipeWaitNs in tc.cuh

fkv_status cache_write(const void* k, const void* v, const int64_t* slot_mapping, int32_t n_tokens,
                       fkv_layer_cache cache, const float* k_scale, const float* v_scale, fkv_scale_gran gran,
                       int32_t layer, const uint8_t* skip_layer_mask, int32_t num_layers, int32_t* fault,
                       fkv_stream_t stream, unsigned long long* clips) {
  if (n_tokens < 0) return FKV_INVALID_ARG;
  if (cache.block_size != 16) return cache.block_size > 0 ? FKV_UNSUPPORTED : FKV_INVALID_ARG;
  if (cache.num_blocks <= 0 || cache.num_kv_heads <= 0 || !valid_format(cache)) return FKV_INVALID_ARG;
  if (!supported_head_dim(cache.head_dim)) return FKV_UNSUPPORTED;
  if (gran != FKV_SCALE_PER_TENSOR && gran != FKV_SCALE_PER_HEAD) return FKV_INVALID_ARG;
  fkv_status st = FKV_OK;
  const bool bf16 = layer_is_bf16(layer, skip_layer_mask, num_layers, &st);
  if (st != FKV_OK) return st;
  if (n_tokens == 0) return FKV_OK;
  if (!k || !v || !slot_mapping || !cache.k_cache || !cache.v_cache) return FKV_INVALID_ARG;
  if (!bf16 && (!k_scale || !v_scale)) return FKV_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(cache.k_cache, 16) || !aligned(cache.v_cache, 16) ||
      !aligned(slot_mapping, 8) || !aligned(clips, 8))
    return FKV_INVALID_ARG;
  return from_cuda(fkv::launch_kv_quant_cache(k, v, slot_mapping, n_tokens, cache, k_scale, v_scale,
                                              gran == FKV_SCALE_PER_HEAD, bf16, fault,
                                              reinterpret_cast<cudaStream_t>(stream), current_num_sms(), clips));
}

}  // namespace

namespace fkv {

// fp8_decode_attn, and with k_new / v_new given fp8_decode_step (the current token written
// into the pools by the same launch).  With `scratch` non-null the workspace arguments are
// ignored: after every argument check and the split-K plan, scratch(need, ...) supplies the
// workspace (fp8_decode_attn_noalloc), so both entry points return the same status for
// the same arguments.
fkv_status decode_entry(const void* k_new, const void* v_new, const void* q, int32_t batch, int32_t num_q_heads,
                        fkv_layer_cache cache, const int32_t* block_table, int32_t max_blocks,
                        const int32_t* context_lens, const float* q_scale, const float* k_scale,
                        const float* v_scale, fkv_scale_gran gran, float softmax_scale, int32_t window,
                        int32_t layer, const uint8_t* skip_layer_mask, int32_t num_layers, void* out,
                        void* workspace, size_t workspace_bytes, ScratchProvider scratch, int32_t num_splits,
                        int32_t* fault, fkv_stream_t stream) {
  const bool step = k_new != nullptr || v_new != nullptr;
  if (batch < 0 || num_q_heads <= 0 || max_blocks <= 0 || window < 0 || num_splits < 0)
    return FKV_INVALID_ARG;
  if (cache.block_size != 16) return cache.block_size > 0 ? FKV_UNSUPPORTED : FKV_INVALID_ARG;
  if (cache.num_blocks <= 0 || cache.num_kv_heads <= 0 || !valid_format(cache)) return FKV_INVALID_ARG;
  if (num_q_heads % cache.num_kv_heads != 0) return FKV_INVALID_ARG;
  if (!supported_head_dim(cache.head_dim)) return FKV_UNSUPPORTED;
  const int G = num_q_heads / cache.num_kv_heads;
  if (!supported_group(G, cache.head_dim)) return FKV_UNSUPPORTED;
  if (gran != FKV_SCALE_PER_TENSOR && gran != FKV_SCALE_PER_HEAD) return FKV_INVALID_ARG;
  if (!(softmax_scale >= 0.f) || std::isinf(softmax_scale)) return FKV_INVALID_ARG;
  if (batch > 65535 || cache.num_kv_heads > 65535) return FKV_UNSUPPORTED;
  fkv_status st = FKV_OK;
  const bool bf16 = layer_is_bf16(layer, skip_layer_mask, num_layers, &st);
  if (st != FKV_OK) return st;
  const int elt = layer_elt(bf16, cache);
  if (batch == 0) return FKV_OK;
  if (step && (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16))) return FKV_INVALID_ARG;
  if (!q || !out || !block_table || !context_lens || !cache.k_cache || !cache.v_cache || (!workspace && !scratch))
    return FKV_INVALID_ARG;
  if (!bf16 && (!q_scale || !k_scale || !v_scale)) return FKV_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(cache.k_cache, 16) || !aligned(cache.v_cache, 16) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4))
    return FKV_INVALID_ARG;
  DecodePlan plan;
  if (!plan_decode(batch, num_q_heads, cache.num_kv_heads, cache.head_dim, max_blocks, window, num_splits, &plan))
    return FKV_UNSUPPORTED;
  const size_t need = plan.o_bytes + plan.lse_bytes + plan.cnt_bytes;
  if (scratch) {
    const fkv_status sst = scratch(need, plan.cnt_bytes, reinterpret_cast<cudaStream_t>(stream), &workspace,
                                   &workspace_bytes);
    if (sst != FKV_OK) return sst;
  }
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return FKV_INVALID_ARG;

  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const uint8_t*>(cache.k_cache);
  p.v_cache = static_cast<const uint8_t*>(cache.v_cache);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.per_head = gran == FKV_SCALE_PER_HEAD;
  p.B = batch;
  p.Hq = num_q_heads;
  p.Hkv = cache.num_kv_heads;
  p.num_blocks = cache.num_blocks;
  p.max_blocks = max_blocks;
  const float tau = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(cache.head_dim));
  p.sm_scale_log2 = tau * 1.4426950408889634f;
  p.window = window;
  p.bps = plan.bps;
  p.max_splits = plan.max_splits;
  // workspace: the split-completion counters first (zero between calls), then the
  // splits' log-sum-exps and normalised outputs (written before they are read)
  p.done = static_cast<int32_t*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.cnt_bytes);
  p.o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.cnt_bytes + plan.lse_bytes);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.fault = fault;
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  const unsigned long long wait_ns = g_decode_wait_ns.load(std::memory_order_relaxed);
  p.pipe_wait_ns = wait_ns != 0 ? wait_ns : kDefaultPipeWaitNs;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fkv::decode_uses_tensor_cores(cache.head_dim, elt)) return from_cuda(fkv::launch_decode_tc(p, cache.head_dim, G, s));
  return from_cuda(fkv::launch_decode(p, cache.head_dim, elt, G, s));
}

}  // namespace fkv

using fkv::decode_entry;

extern "C" {

const char* fkv_status_string(fkv_status status) {
  switch (status) {
    case FKV_OK: return "ok";
    case FKV_INVALID_ARG: return "invalid argument";
    case FKV_UNSUPPORTED: return "unsupported";
    case FKV_CUDA_ERROR: return "cuda error";
  }
  return "unknown status";
}

int32_t fkv_version(void) { return 105; }

void fkv_set_decode_wait_limit_ns(unsigned long long ns) { g_decode_wait_ns.store(ns, std::memory_order_relaxed); }


fkv_status kv_quant_cache(const void* k, const void* v, const int64_t* slot_mapping, int32_t n_tokens,
                          fkv_layer_cache cache, const float* k_scale, const float* v_scale,
                          fkv_scale_gran gran, int32_t layer, const uint8_t* skip_layer_mask,
                          int32_t num_layers, int32_t* fault, fkv_stream_t stream) {
  return cache_write(k, v, slot_mapping, n_tokens, cache, k_scale, v_scale, gran, layer, skip_layer_mask, num_layers,
                     fault, stream, nullptr);
}

fkv_status kv_quant_cache_clips(const void* k, const void* v, const int64_t* slot_mapping, int32_t n_tokens,
                                fkv_layer_cache cache, const float* k_scale, const float* v_scale,
                                fkv_scale_gran gran, int32_t layer, const uint8_t* skip_layer_mask,
                                int32_t num_layers, unsigned long long* clip_counts, int32_t* fault,
                                fkv_stream_t stream) {
  if (clip_counts == nullptr) return FKV_INVALID_ARG;
  return cache_write(k, v, slot_mapping, n_tokens, cache, k_scale, v_scale, gran, layer, skip_layer_mask, num_layers,
                     fault, stream, clip_counts);
}

size_t fp8_decode_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t max_blocks, int32_t window,
                                      int32_t num_splits) {
  DecodePlan plan;
  if (!supported_head_dim(head_dim)) return 0;
  if (!plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, window, num_splits, &plan)) return 0;
  return plan.o_bytes + plan.lse_bytes + plan.cnt_bytes;
}

int32_t fp8_decode_attn_split_blocks(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_blocks, int32_t window,
                                     int32_t num_splits) {
  DecodePlan plan;
  if (!plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, window, num_splits, &plan)) return 0;
  return plan.bps;
}

int32_t fkv_decode_block_n(int32_t head_dim, int32_t layer_kind) {
  const int elt = layer_kind == 0 ? 1 : layer_kind == 1 ? 2 : layer_kind == 2 ? 3 : 0;
  return elt != 0 && fkv::decode_uses_tensor_cores(head_dim, elt) ? 16 * decode_tile_blocks(head_dim) : 0;
}

int32_t fp8_decode_attn_num_splits(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_blocks, int32_t window,
                                   int32_t num_splits) {
  DecodePlan plan;
  if (!plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, window, num_splits, &plan)) return 0;
  return plan.max_splits;
}

fkv_status fp8_decode_attn(const void* q, int32_t batch, int32_t num_q_heads, fkv_layer_cache cache,
                           const int32_t* block_table, int32_t max_blocks, const int32_t* context_lens,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           fkv_scale_gran gran, float softmax_scale, int32_t window, int32_t layer,
                           const uint8_t* skip_layer_mask, int32_t num_layers, void* out, void* workspace,
                           size_t workspace_bytes, int32_t num_splits, int32_t* fault,
                           fkv_stream_t stream) {
  return decode_entry(nullptr, nullptr, q, batch, num_q_heads, cache, block_table, max_blocks, context_lens, q_scale,
                      k_scale, v_scale, gran, softmax_scale, window, layer, skip_layer_mask, num_layers, out, workspace,
                      workspace_bytes, nullptr, num_splits, fault, stream);
}

fkv_status fp8_decode_step(const void* k_new, const void* v_new, const void* q, int32_t batch,
                           int32_t num_q_heads, fkv_layer_cache cache, const int32_t* block_table,
                           int32_t max_blocks, const int32_t* context_lens, const float* q_scale,
                           const float* k_scale, const float* v_scale, fkv_scale_gran gran,
                           float softmax_scale, int32_t window, int32_t layer, const uint8_t* skip_layer_mask,
                           int32_t num_layers, void* out, void* workspace, size_t workspace_bytes,
                           int32_t num_splits, int32_t* fault, fkv_stream_t stream) {
  if (!k_new || !v_new) return FKV_INVALID_ARG;
  return decode_entry(k_new, v_new, q, batch, num_q_heads, cache, block_table, max_blocks, context_lens, q_scale,
                      k_scale, v_scale, gran, softmax_scale, window, layer, skip_layer_mask, num_layers, out, workspace,
                      workspace_bytes, nullptr, num_splits, fault, stream);
}

int32_t fkv_prefill_block_n(int32_t head_dim) { return supported_head_dim(head_dim) ? 128 : 0; }

fkv_status fp8_prefill_attn(const void* q, const int32_t* cu_seqlens_q, int32_t batch, int32_t num_q_heads,
                            int32_t max_q_len, fkv_layer_cache cache, const int32_t* block_table,
                            int32_t max_blocks, const int32_t* context_lens, const float* q_scale,
                            const float* k_scale, const float* v_scale, fkv_scale_gran gran,
                            float softmax_scale, int32_t causal, int32_t window, int32_t promote_every,
                            int32_t layer, const uint8_t* skip_layer_mask, int32_t num_layers, void* out,
                            int32_t* fault, fkv_stream_t stream) {
  if (batch < 0 || num_q_heads <= 0 || max_q_len < 0 || max_blocks <= 0) return FKV_INVALID_ARG;
  if (cache.block_size != 16) return cache.block_size > 0 ? FKV_UNSUPPORTED : FKV_INVALID_ARG;
  if (cache.num_blocks <= 0 || cache.num_kv_heads <= 0 || !valid_format(cache)) return FKV_INVALID_ARG;
  if (num_q_heads % cache.num_kv_heads != 0) return FKV_INVALID_ARG;
  if (!supported_head_dim(cache.head_dim)) return FKV_UNSUPPORTED;
  if (gran != FKV_SCALE_PER_TENSOR && gran != FKV_SCALE_PER_HEAD) return FKV_INVALID_ARG;
  if (!(softmax_scale >= 0.f) || std::isinf(softmax_scale)) return FKV_INVALID_ARG;
  if (window < 0 || promote_every < 0) return FKV_INVALID_ARG;
  if (window > 0 && !causal) return FKV_UNSUPPORTED;                        // a window is causal
  fkv_status st = FKV_OK;
  const bool bf16 = layer_is_bf16(layer, skip_layer_mask, num_layers, &st);
  if (st != FKV_OK) return st;
  // bf16 layers at head_dim 256: TMEM holds one 128-column O_tile
  if (promote_every >= 2 && cache.head_dim > 128 && bf16) return FKV_UNSUPPORTED;
  if (!bf16 && cache.kv_format == FKV_KV_E5M2) return FKV_UNSUPPORTED;  // e5m2 layers: decode only
  if (batch > 65535 || num_q_heads > 65535) return FKV_UNSUPPORTED;
  if (batch == 0 || max_q_len == 0) return FKV_OK;
  if (!q || !cu_seqlens_q || !block_table || !context_lens || !cache.k_cache || !cache.v_cache || !out)
    return FKV_INVALID_ARG;
  if (!bf16 && (!q_scale || !k_scale || !v_scale)) return FKV_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(cache.k_cache, 16) || !aligned(cache.v_cache, 16) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4) || !aligned(cu_seqlens_q, 4))
    return FKV_INVALID_ARG;
  fkv::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.cu_q = cu_seqlens_q;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.per_head = gran == FKV_SCALE_PER_HEAD;
  p.B = batch;
  p.Hq = num_q_heads;
  p.Hkv = cache.num_kv_heads;
  p.num_blocks = cache.num_blocks;
  p.max_blocks = max_blocks;
  p.n_qtiles = (max_q_len + 127) / 128;
  const float tau = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(cache.head_dim));
  p.sm_scale_log2 = tau * 1.4426950408889634f;
  p.causal = causal != 0;
  p.promote_every = promote_every;
  p.window = window;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.fault = fault;
  return from_cuda(fkv::launch_prefill(p, cache.head_dim, bf16, cache.k_cache, cache.v_cache,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
