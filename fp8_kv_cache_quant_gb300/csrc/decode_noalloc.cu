// fp8_decode_attn_noalloc: the split-K decode of fp8_decode_attn with its scratch held in
// a fixed device array of this library instead of a caller-supplied workspace.
//
// Some callers cannot hand the library a workspace: a host framework whose memory pool
// owns the whole device and gives plugins only their input and output pointers, or a
// serving loop that must not call cudaMalloc/cudaFree because those calls can
// synchronise the device and stall every stream.  For them this entry point keeps the
// split partials in the file-scope array below, sized once for every GPU that loads the
// library, and allocates nothing itself.
#include <mutex>

#include "common.cuh"

namespace {

// Scratch for the split partials (o / l and log-sum-exp of every split).  Every call on
// a device reuses the same bytes; each call writes every partial it later reads, so no
// part of it has to start at zero.
static __device__ __align__(256) unsigned char g_decode_scratch[FKV_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The name of the array is
// only a host-side stand-in; the address is looked up once per device, with that device
// current, and cached.
fkv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FKV_CUDA_ERROR;
  }
  if (dev < 0 || dev >= kMaxDevices) return FKV_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FKV_CUDA_ERROR;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FKV_OK;
}

}  // namespace

extern "C" fkv_status fp8_decode_attn_noalloc(
    const void* q, int32_t batch, int32_t num_q_heads, fkv_layer_cache cache, const int32_t* block_table,
    int32_t max_blocks, const int32_t* context_lens, const float* q_scale, const float* k_scale,
    const float* v_scale, fkv_scale_gran gran, float softmax_scale, int32_t window, int32_t layer,
    const uint8_t* skip_layer_mask, int32_t num_layers, void* out, int32_t num_splits, int32_t* fault,
    fkv_stream_t stream) {
  if (batch < 0 || num_q_heads <= 0 || cache.num_kv_heads <= 0 || max_blocks <= 0) return FKV_INVALID_ARG;
  if (batch == 0) return FKV_OK;
  const size_t need = fp8_decode_attn_workspace_size(batch, num_q_heads, cache.num_kv_heads, cache.head_dim,
                                                     max_blocks, window, num_splits);
  if (need == 0) {
    // sizes the split-K plan rejects: let the regular entry point report why
    return fp8_decode_attn(q, batch, num_q_heads, cache, block_table, max_blocks, context_lens, q_scale, k_scale,
                           v_scale, gran, softmax_scale, window, layer, skip_layer_mask, num_layers, out, nullptr,
                           0, num_splits, fault, stream);
  }
  if (need > static_cast<size_t>(FKV_NOALLOC_WORKSPACE_BYTES)) return FKV_INVALID_ARG;  // beyond the fixed scratch
  void* ws = nullptr;
  const fkv_status st = scratch_address(&ws);
  if (st != FKV_OK) return st;
  return fp8_decode_attn(q, batch, num_q_heads, cache, block_table, max_blocks, context_lens, q_scale, k_scale,
                         v_scale, gran, softmax_scale, window, layer, skip_layer_mask, num_layers, out, ws,
                         static_cast<size_t>(FKV_NOALLOC_WORKSPACE_BYTES), num_splits, fault, stream);
}
