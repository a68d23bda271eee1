// Internal launcher interfaces between the C ABI (abi.cu) and the kernel files.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/fp8kv.h"

namespace fkv {

// Pool blocks per decode split, at most (the CUDA-core decode and the tensor-core decode at
// head_dim 128 and 256 stage a split's block ids in shared memory).
constexpr int kMaxSplitBlocks = 256;

struct DecodeParams {
  const __nv_bfloat16* q;      // [B][Hq][D]
  const uint8_t* k_cache;      // pool bytes
  const uint8_t* v_cache;
  const int32_t* block_table;  // [B][max_blocks]
  const int32_t* context_lens; // [B]
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int per_head;
  int B, Hq, Hkv, num_blocks, max_blocks;
  float sm_scale_log2;  // softmax_scale * log2(e)
  int window;
  int bps;              // blocks per split
  int max_splits;
  float* o_part;        // [B][Hq][max_splits][D]
  float* lse_part;      // [B][Hq][max_splits], base 2
  int32_t* done;        // [B][Hkv] splits finished (zeroed before the launch)
  __nv_bfloat16* out;   // [B][Hq][D]
  int32_t* fault;
  // the current token's K and V, bf16 [B][Hkv][D], quantised into the (e4m3) pools at
  // position T - 1 by the launch itself (fp8_decode_step); null: the pools are complete
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  // wall-clock bound of the tensor-core decode's pipeline waits (ns); the waits that let
  // issued copies and products drain before the CTA exits keep their own bound
  uint64_t pipe_wait_ns;
};

struct PrefillParams {
  const __nv_bfloat16* q;       // [total_q][Hq][D]
  const int32_t* cu_q;          // [B + 1]
  const int32_t* block_table;   // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int per_head;
  int B, Hq, Hkv, num_blocks, max_blocks, n_qtiles;
  float sm_scale_log2;
  int causal;
  int promote_every;            // 1: every tile; N >= 2: every N tiles; 0: never
  int window;                   // 0 = full, else the last `window` keys of each query
  __nv_bfloat16* out;           // [total_q][Hq][D]
  int32_t* fault;
};

cudaError_t launch_prefill(const PrefillParams& p, int D, bool bf16_layer, void* k_cache, void* v_cache,
                           cudaStream_t s);

// Launch `kern` with programmatic stream serialisation (the kernel must call griddep_wait
// before touching global memory that earlier kernels produce or consume).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

cudaError_t launch_kv_quant_cache(const void* k, const void* v, const int64_t* slots, int n_tokens,
                                  const fkv_layer_cache& cache, const float* ks, const float* vs,
                                  int per_head, bool bf16_layer, int32_t* fault, cudaStream_t s,
                                  int num_sms, unsigned long long* clips);

// elt: the pool's element type, 1 e4m3, 2 bf16, 3 e5m2
cudaError_t launch_decode(const DecodeParams& p, int D, int elt, int G, cudaStream_t s);

// e4m3 layers (elt 1, head_dim 64 / 128 / 256) decode on the tensor cores (FP8 P, 128-key
// tiles); bf16 and e5m2 layers on the CUDA cores (P exact).
bool decode_uses_tensor_cores(int D, int elt);
cudaError_t launch_decode_tc(const DecodeParams& p, int D, int G, cudaStream_t s);

// Supplies the decode's workspace of `need` bytes when the caller passes none: sets *ws
// (256-byte aligned) and *bytes, with its first `counter_bytes` (the split counters) zero
// by the time work enqueued afterwards on `stream` runs, or returns the status the entry
// point then returns.
using ScratchProvider = fkv_status (*)(size_t need, size_t counter_bytes, cudaStream_t stream, void** ws,
                                       size_t* bytes);

// The whole of fp8_decode_attn (k_new = v_new = NULL) and fp8_decode_step: argument
// checks, the split-K plan, then the launch.  With scratch non-null the workspace comes
// from it, after every check (fp8_decode_attn_noalloc).
fkv_status decode_entry(const void* k_new, const void* v_new, const void* q, int32_t batch, int32_t num_q_heads,
                        fkv_layer_cache cache, const int32_t* block_table, int32_t max_blocks,
                        const int32_t* context_lens, const float* q_scale, const float* k_scale,
                        const float* v_scale, fkv_scale_gran gran, float softmax_scale, int32_t window,
                        int32_t layer, const uint8_t* skip_layer_mask, int32_t num_layers, void* out,
                        void* workspace, size_t workspace_bytes, ScratchProvider scratch, int32_t num_splits,
                        int32_t* fault, fkv_stream_t stream);

}  // namespace fkv
