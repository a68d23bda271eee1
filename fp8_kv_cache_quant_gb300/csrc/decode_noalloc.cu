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

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace {

// Scratch for the split-completion counters (at its start) and the split partials (o / l
// and log-sum-exp of every split).  Every call on a device reuses the same bytes: device
// arrays start zero-filled, each call returns the counters to zero, and each split writes
// every partial that the merge later reads.
static __device__ __align__(256) unsigned char g_decode_scratch[FKV_NOALLOC_WORKSPACE_BYTES];

// The array's device address belongs to the context the module was loaded into: the
// primary context of a device until a device reset destroys it, or a context the caller
// created and made current.  The address is therefore cached per context, keyed by the
// driver's context id (unique for the life of the process, never reused after a reset),
// and looked up with cudaGetSymbolAddress, with that context current, the first time a
// context calls.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct Cached {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kMaxContexts = 64;
std::mutex g_mu;
Cached g_cache[kMaxContexts];
int g_cached = 0;
CtxGetCurrentFn g_get_current = nullptr;
CtxGetIdFn g_get_id = nullptr;
bool g_driver_looked_up = false;

template <typename Fn>
Fn driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<Fn>(ptr);
}

fkv_status noalloc_address(void** ws, size_t* bytes);

// Id of the current context, or false when the driver cannot tell (no context current).
bool current_ctx_id(unsigned long long* id) {
  CUcontext ctx = nullptr;
  if (!g_get_current || !g_get_id || g_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_get_id(ctx, id) == CUDA_SUCCESS;
}

// Supplies fp8_decode_attn's workspace from the fixed array (a ScratchProvider): sizes
// beyond the array are FKV_INVALID_ARG.  The split counters at the array's start are
// cleared on the stream first: an earlier call with fewer (sequence, KV head) units left
// other scratch where this call's counters lie, and the array cannot be handed to the
// caller to clear.
fkv_status noalloc_scratch(size_t need, size_t counter_bytes, cudaStream_t stream, void** ws, size_t* bytes) {
  if (need > static_cast<size_t>(FKV_NOALLOC_WORKSPACE_BYTES)) return FKV_INVALID_ARG;
  const fkv_status st = noalloc_address(ws, bytes);
  if (st != FKV_OK) return st;
  if (cudaMemsetAsync(*ws, 0, counter_bytes, stream) != cudaSuccess) return FKV_CUDA_ERROR;
  return FKV_OK;
}

// The array's device address in the current context (looked up on the context's first call).
fkv_status noalloc_address(void** ws, size_t* bytes) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_driver_looked_up) {
    g_get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    g_get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    g_driver_looked_up = true;
  }
  unsigned long long id = 0;
  bool have_id = current_ctx_id(&id);
  if (have_id) {
    for (int i = 0; i < g_cached; ++i)
      if (g_cache[i].ctx_id == id) {
        *ws = g_cache[i].addr;
        *bytes = FKV_NOALLOC_WORKSPACE_BYTES;
        return FKV_OK;
      }
  }
  // first call in this context: the lookup also makes the runtime's primary context
  // current when none was (the module is loaded into it)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return FKV_CUDA_ERROR;
  }
  if (!have_id) have_id = current_ctx_id(&id);
  if (have_id && g_cached < kMaxContexts) g_cache[g_cached++] = Cached{id, p};
  *ws = p;
  *bytes = FKV_NOALLOC_WORKSPACE_BYTES;
  return FKV_OK;
}

}  // namespace

extern "C" fkv_status fp8_decode_attn_noalloc(
    const void* q, int32_t batch, int32_t num_q_heads, fkv_layer_cache cache, const int32_t* block_table,
    int32_t max_blocks, const int32_t* context_lens, const float* q_scale, const float* k_scale,
    const float* v_scale, fkv_scale_gran gran, float softmax_scale, int32_t window, int32_t layer,
    const uint8_t* skip_layer_mask, int32_t num_layers, void* out, int32_t num_splits, int32_t* fault,
    fkv_stream_t stream) {
  return fkv::decode_entry(nullptr, nullptr, q, batch, num_q_heads, cache, block_table, max_blocks, context_lens,
                           q_scale, k_scale, v_scale, gran, softmax_scale, window, layer, skip_layer_mask,
                           num_layers, out, nullptr, 0, noalloc_scratch, num_splits, fault, stream);
}
