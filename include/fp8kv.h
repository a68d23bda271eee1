/*
 * fp8kv — FP8 (e4m3) KV-cache quantisation and FP8 attention for GB300 (sm_103a).
 *
 * C ABI of libfp8kv.so.  Every tensor argument is a plain device pointer owned by the
 * caller; the library allocates nothing, keeps no state between calls (the exceptions:
 * the one fixed device array that is the scratch of fp8_decode_attn_noalloc, and the wait
 * bound of the test hook fkv_set_decode_wait_limit_ns), and enqueues its kernels on the
 * given stream without synchronising.  Host pointers are marked "host".
 *
 * The operations restate the vLLM blog "FP8 KV-Cache and Attention quantization in
 * vLLM" (2026-04-22):
 *   - 引言: `--kv-cache-dtype fp8` stores K/V in e4m3 and runs the whole attention in
 *     FP8, the QK and Score*V matrix products included;
 *   - "Kernel 与 vLLM 改进": two-level accumulation (partial sums promoted into a true
 *     FP32 register), skip layers (`--kv-cache-dtype-skip-layers sliding_window` keeps
 *     sliding-window layers in BF16), per-head scales (one scale per KV head, also for
 *     the cache write `reshape_and_cache_flash`), query quantisation, decode-tuned
 *     configurations;
 *   - "大 Head Dimension 的限制": promoting every N steps or never (prefill).
 *
 * Formats and layouts (fixed by this library; the pages are silent on them):
 *   e4m3      FP8 E4M3 "fn": 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no
 *             infinities, S.1111.111 = NaN, largest finite +-448.  Quantisation of x
 *             with scale s is e4m3(fl32(x * fl32(1/s))), round-to-nearest-even,
 *             saturating; dequantisation is code * s.
 *   K/V pool  per layer, [num_blocks][num_kv_heads][block_size][head_dim], one byte per
 *             element (e4m3) or two (bf16, skip layers); block_size must be 16.
 *   positions token position p of sequence b lives in slot
 *             block_table[b][p / 16] * 16 + p % 16.
 *   scales    float32 device arrays.  FKV_SCALE_PER_TENSOR: q/k/v scale arrays hold one
 *             value.  FKV_SCALE_PER_HEAD: k/v scales hold num_kv_heads values and the
 *             query scale num_q_heads values.
 *   GQA       query head h reads KV head h / (num_q_heads / num_kv_heads).
 *
 * Launches.  The decode kernels are launched with programmatic stream serialisation: a
 * decode kernel may be scheduled while the kernel before it in the stream finishes, and
 * sets up its barriers and tensor memory then, but reads and writes no global memory
 * until that kernel has completed, so the stream's ordering is kept.
 *
 * Errors.  Argument checks run on the host before anything is enqueued and return
 * FKV_INVALID_ARG or FKV_UNSUPPORTED; a failed launch returns FKV_CUDA_ERROR.  Data
 * errors that only the GPU can see (a block id outside [0, num_blocks), a slot outside
 * the pool, a context longer than the block table, a prefill chunk longer than its
 * context, a pipeline wait that ran out of time) never trap: the kernel skips or
 * clamps the access and ORs an FKV_FAULT_* bit into *fault (a caller-owned device
 * int32, may be NULL).  Kernels never spin without a time bound.
 */
#ifndef FP8KV_H
#define FP8KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* fkv_stream_t;

typedef enum {
  FKV_OK = 0,
  FKV_INVALID_ARG = 1,  /* NULL pointer, negative size, misaligned pointer, ...      */
  FKV_UNSUPPORTED = 2,  /* valid but not implemented (head_dim, group size, ...)    */
  FKV_CUDA_ERROR = 3    /* a CUDA call or kernel launch failed                      */
} fkv_status;

typedef enum {
  FKV_SCALE_PER_TENSOR = 0, /* one scale for Q, one for K, one for V                 */
  FKV_SCALE_PER_HEAD = 1    /* K/V: one per KV head; Q: one per query head           */
} fkv_scale_gran;

/* Bits ORed into the caller's device fault word. */
#define FKV_FAULT_BLOCK_ID 1 /* block table entry outside [0, num_blocks): block 0 read instead */
#define FKV_FAULT_SLOT 2     /* cache-write slot >= num_blocks * block_size: token skipped      */
#define FKV_FAULT_CONTEXT 4  /* context length < 0 or > max_blocks * block_size: clamped      */
#define FKV_FAULT_TIMEOUT 8  /* an in-kernel wait ran out of time (200 ms per pipeline wait in the
                                tensor-core kernels, 1 s elsewhere): the CTA's remaining work is
                                abandoned after its copies and products drain; its partial
                                results are undefined                                             */
#define FKV_FAULT_QLEN 16    /* prefill: query length > context length: sequence skipped     */
#define FKV_FAULT_WORKSPACE 32 /* decode: a split counter of the workspace was not zero when the
                                  call began (zero-fill a workspace before its first call)     */

/* FP8 format of a layer's pools (fkv_layer_cache.kv_format). */
typedef enum {
  FKV_KV_E4M3 = 0, /* e4m3 "fn": the format of the FP8 attention (default) */
  FKV_KV_E5M2 = 1  /* e5m2 (vLLM's other FP8 KV-cache format): dequantised, attended in bf16 precision */
} fkv_kv_format;

/* One layer of the paged cache.  k_cache / v_cache: device pools, 16-byte aligned,
 * [num_blocks][num_kv_heads][block_size][head_dim] of FP8 codes (1 byte, format
 * kv_format) or bf16 (2 bytes): a layer named by the skip-layer mask is bf16 whatever
 * kv_format says. */
typedef struct {
  void* k_cache;
  void* v_cache;
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t kv_format; /* fkv_kv_format */
} fkv_layer_cache;

/* Human-readable name of a status code (static string). */
const char* fkv_status_string(fkv_status status);

/* Library ABI version (major * 100 + minor). */
int32_t fkv_version(void);

/*
 * fkv_set_decode_wait_limit_ns — test hook for the timeout path of the tensor-core decode.
 *
 * Sets, for fp8_decode_attn / fp8_decode_step / fp8_decode_attn_noalloc launches on e4m3
 * layers made after the call (process-wide), the wall-clock bound of each in-kernel
 * pipeline wait; 0 restores the default of 200 ms.  A bound shorter than the pipeline's
 * own latency makes the first unsatisfied wait run out, so that FKV_FAULT_TIMEOUT and the
 * recovery that follows can be exercised without a stalled GPU: the CTA stops, lets
 * every copy and product it issued complete (those waits keep the 200 ms bound), frees
 * its tensor memory and returns; the output of such a launch is undefined (the split
 * merge reads whatever the workspace held).  Not for production use.
 */
void fkv_set_decode_wait_limit_ns(unsigned long long ns);

/*
 * kv_quant_cache — write new tokens' K and V into one layer of the paged cache.
 *
 * The blog's cache write (`reshape_and_cache_flash`, section "Kernel 与 vLLM 改进",
 * paragraph "Per-Head Scales") extended to a per-KV-head scale array; skip layers
 * ("跳过 Layer") are stored as an exact bf16 copy.
 *
 *   k, v          device bf16 [n_tokens][num_kv_heads][head_dim], contiguous, 16-byte aligned
 *   slot_mapping  device int64 [n_tokens]; slot = block * 16 + offset; a negative slot
 *                 skips the token (padding); a slot beyond the pool raises FKV_FAULT_SLOT
 *   cache         the layer's pools (see fkv_layer_cache)
 *   k_scale, v_scale  device float32 [1] or [num_kv_heads] (per gran); unused for
 *                 skip layers (may be NULL there)
 *   layer, skip_layer_mask (host uint8 [num_layers], may be NULL = no skipped layer),
 *   num_layers    skip_layer_mask[layer] != 0 selects the bf16 pool format
 *   fault         device int32 or NULL
 * Each element is e4m3(fl32(x * fl32(1/scale))) (round-to-nearest-even, saturating;
 * e5m2 likewise on pools with cache.kv_format FKV_KV_E5M2, saturating to +-57344); every
 * other byte of the pools keeps its value.
 */
fkv_status kv_quant_cache(const void* k, const void* v, const int64_t* slot_mapping,
                          int32_t n_tokens, fkv_layer_cache cache, const float* k_scale,
                          const float* v_scale, fkv_scale_gran gran, int32_t layer,
                          const uint8_t* skip_layer_mask, int32_t num_layers,
                          int32_t* fault, fkv_stream_t stream);

/*
 * kv_quant_cache_clips — kv_quant_cache that also counts clipped elements.
 *
 * The KV-cache quantisation explainer's pre-production checklist asks for the clipping
 * frequency where it can be observed.  Same write as kv_quant_cache; in addition
 * clip_counts[0] and clip_counts[1] (device uint64, accumulated atomically; the caller
 * zeroes them) grow by the number of K and V elements whose scaled value
 * fl32(x * fl32(1/scale)) lies beyond the format's largest finite value (448 for
 * e4m3, 57344 for e5m2) and is therefore clipped (NaN is not counted; skip layers clip
 * nothing).  clip_counts NULL or not 8-byte aligned:
 * FKV_INVALID_ARG.
 */
fkv_status kv_quant_cache_clips(const void* k, const void* v, const int64_t* slot_mapping,
                                int32_t n_tokens, fkv_layer_cache cache, const float* k_scale,
                                const float* v_scale, fkv_scale_gran gran, int32_t layer,
                                const uint8_t* skip_layer_mask, int32_t num_layers,
                                unsigned long long* clip_counts, int32_t* fault, fkv_stream_t stream);

/*
 * Workspace bytes fp8_decode_attn needs for these sizes (same argument meaning as
 * there).  Returns 0 for invalid sizes.
 */
size_t fp8_decode_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t max_blocks, int32_t window,
                                      int32_t num_splits);

/* Number of context splits per sequence fp8_decode_attn uses for these sizes. */
int32_t fp8_decode_attn_num_splits(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_blocks, int32_t window,
                                   int32_t num_splits);

/*
 * Pool blocks per context split of fp8_decode_attn for these sizes (a multiple of u,
 * the blocks of one tensor-core decode tile: u = 16 at head_dim 64, else 8): split s of
 * a sequence covers blocks [lo / 16 + s * n, lo / 16 + (s + 1) * n).  0 for invalid
 * sizes.  With n_blk = max_blocks (window 0) or min(max_blocks, ceil(window / 16) + 1), a
 * requested num_splits > 0 gives ceil(n_blk / num_splits) blocks, at most 256 and at
 * least ceil(n_blk / 1024), rounded up to a multiple of u (a result above 256 means the
 * context is too long: 0).  num_splits 0 picks, among the multiples of u up to 256, the
 * count c minimising waves(c) * min(c, n_blk), where waves(c) = ceil(batch *
 * num_kv_heads * ceil(n_blk / c) / (3 * SMs of the current device)); ties go to the
 * larger c.
 */
int32_t fp8_decode_attn_split_blocks(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_blocks, int32_t window,
                                     int32_t num_splits);

/*
 * Keys per tile over which fp8_decode_attn rounds P to e4m3 for a layer of this head_dim
 * and kind (0: e4m3 pools, 1: a skip layer's bf16 pools, 2: e5m2 pools), or 0 when that
 * layer's decode keeps P exact.  Tiles start at each split's first block.
 */
int32_t fkv_decode_block_n(int32_t head_dim, int32_t layer_kind);

/*
 * fp8_decode_attn — one decode step of paged GQA attention for one layer.
 *
 * For every sequence b and query head h (KV head g = h / G): keys j in
 * [lo, T_b) with T_b = context_lens[b] (the current token included, already written
 * by kv_quant_cache) and lo = max(0, T_b - window) (window 0 = all keys);
 *   s_j = (e4m3(q*1/q_s) * q_s) . (k8_j * k_s[g]) * softmax_scale,
 *   out = sum_j softmax(s)_j * (v8_j * v_s[g])     (bf16 [batch][num_q_heads][head_dim]).
 * The context is split across CTAs (split-K, the blog's decode-tuned configurations);
 * each split keeps its softmax state and P.V sum in FP32, and the CTA that finishes a
 * (sequence, KV head) last merges the splits through their log-sum-exp in FP32 — the
 * two-level accumulation of the blog's "Two-level accumulation" paragraph, so a 100k+
 * key contraction is summed in true FP32.
 * e4m3 layers (head_dim 64, 128 or 256) run on the tensor cores, FP8 QK and Score*V as
 * in the blog's FP8 attention: S^T = K8 Q8^T and O^T = V8^T P8^T per tile of
 * fkv_decode_block_n keys (128; 256 at head_dim 64) with
 * P8 = e4m3(p * 448) relative to the split's running maximum, the denominator summing
 * the unrounded p, and each tile's partial promoted into FP32 registers.  Skip layers
 * read a bf16 pool, quantise nothing and keep P exact; e5m2 layers (cache.kv_format)
 * dequantise their codes with the scales and attend with the bf16 query and exact P on
 * the CUDA cores.  fkv_decode_block_n tells which applies.
 *
 *   q             device bf16 [batch][num_q_heads][head_dim]
 *   block_table   device int32 [batch][max_blocks]
 *   context_lens  device int32 [batch]
 *   q_scale, k_scale, v_scale  device float32 (see gran); unused on skip layers
 *   softmax_scale 0 selects 1/sqrt(head_dim)
 *   window        0 = full attention, else the number of most recent keys attended
 *   out           device bf16 [batch][num_q_heads][head_dim]
 *   workspace     device, >= fp8_decode_attn_workspace_size(...) bytes, 256-byte aligned,
 *                 zero-filled before its first call.  Its first 4 * batch * num_kv_heads
 *                 bytes are split-completion counters, which must be zero when a call
 *                 begins and which every call leaves at zero; the rest is scratch, written
 *                 before it is read.  A workspace is therefore reused without clearing by
 *                 calls in one stream with the same or a smaller batch * num_kv_heads
 *                 (zero it again when that grows).  A counter found non-zero sets
 *                 FKV_FAULT_WORKSPACE.
 *   num_splits    0 = automatic, else the requested number of context splits (each split
 *                 is then rounded up to whole tiles, see fp8_decode_attn_split_blocks, so
 *                 fewer may result)
 * head_dim in {64, 128, 256}; G = num_q_heads / num_kv_heads in {1, 2, 4, 8, 16} with
 * G * head_dim <= 2048.  A sequence with no key gets a zero row.
 */
fkv_status fp8_decode_attn(const void* q, int32_t batch, int32_t num_q_heads,
                           fkv_layer_cache cache, const int32_t* block_table, int32_t max_blocks,
                           const int32_t* context_lens, const float* q_scale, const float* k_scale,
                           const float* v_scale, fkv_scale_gran gran, float softmax_scale,
                           int32_t window, int32_t layer, const uint8_t* skip_layer_mask,
                           int32_t num_layers, void* out, void* workspace, size_t workspace_bytes,
                           int32_t num_splits, int32_t* fault, fkv_stream_t stream);

/*
 * fp8_decode_step — the current token's cache write and fp8_decode_attn in one launch.
 *
 * A decode step of one layer writes the new token's K and V into the paged cache and
 * then attends over the whole context, the new token included (the blog's cache write
 * reshape_and_cache_flash followed by the decode attention).  For every sequence b with
 * T_b = context_lens[b] >= 1, the rows k_new[b][g][:] and v_new[b][g][:] of every KV
 * head g are written into the pools at position T_b - 1 (block
 * block_table[b][(T_b - 1) / 16], slot (T_b - 1) % 16) exactly as kv_quant_cache writes
 * them — e4m3(fl32(x * fl32(1 / s))) with the same k_scale / v_scale and gran, e5m2 likewise
 * on e5m2 pools, an exact copy on a skip layer's bf16 pools — then the attention is that
 * of fp8_decode_attn with the same arguments.  The write is done by the CTA whose context
 * split holds position T_b - 1, before its copies read that block, so the result equals
 * kv_quant_cache followed by fp8_decode_attn, pool bytes and output bit for bit, with one
 * launch instead of two.
 *
 *   k_new, v_new  device bf16 [batch][num_kv_heads][head_dim], 16-byte aligned
 *   all other arguments as for fp8_decode_attn
 * A block id out of range is reported as for fp8_decode_attn and its row is not written;
 * so is a context length outside [0, max_blocks * 16] (FKV_FAULT_CONTEXT): no pool byte
 * changes.
 */
fkv_status fp8_decode_step(const void* k_new, const void* v_new, const void* q, int32_t batch,
                           int32_t num_q_heads, fkv_layer_cache cache, const int32_t* block_table,
                           int32_t max_blocks, const int32_t* context_lens, const float* q_scale,
                           const float* k_scale, const float* v_scale, fkv_scale_gran gran,
                           float softmax_scale, int32_t window, int32_t layer, const uint8_t* skip_layer_mask,
                           int32_t num_layers, void* out, void* workspace, size_t workspace_bytes,
                           int32_t num_splits, int32_t* fault, fkv_stream_t stream);

/* Size of the fixed device scratch used by fp8_decode_attn_noalloc (16 MiB per GPU). */
#define FKV_NOALLOC_WORKSPACE_BYTES (16u << 20)

/*
 * fp8_decode_attn_noalloc — fp8_decode_attn for callers that cannot provide a workspace.
 *
 * The pages have no counterpart: this is a convenience of this library.  Callers such
 * as plugins inside a framework that owns all device memory, or serving loops that
 * must never call cudaMalloc/cudaFree (both can synchronise the device), get the same
 * computation with the split partials kept in a fixed 16 MiB device array of the
 * library (FKV_NOALLOC_WORKSPACE_BYTES), present on every GPU that loads the library
 * until the process exits.  Arguments mean what they mean for fp8_decode_attn; there is
 * no workspace argument.  Nothing is allocated.
 *
 *   - Returns FKV_INVALID_ARG when fp8_decode_attn_workspace_size(...) for these sizes
 *     exceeds FKV_NOALLOC_WORKSPACE_BYTES (use fp8_decode_attn with a caller workspace
 *     for such sizes), and otherwise exactly the status fp8_decode_attn returns for the
 *     same arguments (the same checks run first, in the same order).
 *   - The first call in a CUDA context (the device's primary context, or a context the
 *     caller made current) looks up the array's device address in that context and
 *     caches it for that context; make that first call before any stream capture.  A
 *     device reset or a new context gets its own lookup on its first call.
 *   - All calls share the one array: calls whose kernels overlap on the GPU (other
 *     streams, other host threads) race on it and produce wrong results.  Calls in one
 *     stream are ordered and safe: each call clears its split counters (the array's
 *     first 4 * batch * num_kv_heads bytes) on the stream before its kernel, and writes
 *     every other scratch byte before it reads it.
 */
fkv_status fp8_decode_attn_noalloc(const void* q, int32_t batch, int32_t num_q_heads,
                                   fkv_layer_cache cache, const int32_t* block_table,
                                   int32_t max_blocks, const int32_t* context_lens,
                                   const float* q_scale, const float* k_scale, const float* v_scale,
                                   fkv_scale_gran gran, float softmax_scale, int32_t window,
                                   int32_t layer, const uint8_t* skip_layer_mask, int32_t num_layers,
                                   void* out, int32_t num_splits, int32_t* fault,
                                   fkv_stream_t stream);

/* Keys per tile of fp8_prefill_attn (its online-softmax and P-rounding granularity). */
int32_t fkv_prefill_block_n(int32_t head_dim);

/*
 * fp8_prefill_attn — FP8 prefill (chunked) attention on tcgen05 tensor cores.
 *
 * Query row i of sequence b (rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1) sits at absolute
 * position p = context_lens[b] - Lq_b + i (the chunk is the tail of the context, its own
 * K/V already written by kv_quant_cache).  With causal != 0 it attends keys [0, p], else
 * all context_lens[b] keys.  Q is quantised to e4m3 in the kernel prologue; S = Q8.K8^T
 * and O_tile = P8.V8 run on the tensor cores with FP32 accumulation in tensor memory;
 * per tile of fkv_prefill_block_n(head_dim) keys the online softmax takes the running
 * max m, P8 = e4m3(exp(s - m) * 448), the denominator sums the unrounded p, and the
 * tile's O partial is promoted into an FP32 accumulator (two-level accumulation).
 * The result is O * v_s / (448 * l) as bf16.
 *
 *   q             device bf16 [total_q][num_q_heads][head_dim] (total_q = cu_seqlens_q[batch])
 *   cu_seqlens_q  device int32 [batch + 1], non-decreasing, starting at 0
 *   max_q_len     host upper bound of every Lq_b (sizes the grid)
 *   causal        non-zero for causal masking
 *   window        0 = full attention; W > 0 keeps, for the row at position p, the keys
 *                 [p - W + 1, p] only (sliding window, causal != 0 required, else
 *                 FKV_UNSUPPORTED; tiles wholly before the CTA's first live key are skipped)
 *   promote_every 1: promote each tile's P.V partial into the FP32 accumulator (two-level
 *                 accumulation, the default); N >= 2: let the tensor core accumulate N tiles
 *                 (rescaled in place when a row's maximum moves) before promoting (at
 *                 head_dim 256 on e4m3 layers only, else FKV_UNSUPPORTED);
 *                 0: never promote — the tensor core accumulates
 *                 the whole contraction (the blog's "大 Head Dimension 的限制": accumulate
 *                 every N steps, or disable two-level accumulation); negative: FKV_INVALID_ARG
 *   out           device bf16 [total_q][num_q_heads][head_dim]
 * e5m2 layers (cache.kv_format FKV_KV_E5M2, not skipped) are FKV_UNSUPPORTED.
 * head_dim in {64, 128, 256}.  Skip (bf16) layers — the layer's bit set in skip_layer_mask —
 * read the bf16 pool and run the same kernel on bf16 operands (kind::f16 MMA, P rounded to
 * bf16, no scales: q_scale/k_scale/v_scale may be NULL); at head_dim 256 their key tiles
 * hold 64 keys (128-key bf16 tiles do not fit in shared memory).
 */
fkv_status fp8_prefill_attn(const void* q, const int32_t* cu_seqlens_q, int32_t batch,
                            int32_t num_q_heads, int32_t max_q_len, fkv_layer_cache cache,
                            const int32_t* block_table, int32_t max_blocks,
                            const int32_t* context_lens, const float* q_scale,
                            const float* k_scale, const float* v_scale, fkv_scale_gran gran,
                            float softmax_scale, int32_t causal, int32_t window,
                            int32_t promote_every, int32_t layer, const uint8_t* skip_layer_mask,
                            int32_t num_layers, void* out, int32_t* fault, fkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_H */
