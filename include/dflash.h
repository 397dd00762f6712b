/*
 * dflash.h -- C ABI of the GB300 (sm_103a) DFlash draft block-attention library.
 *
 * The library computes the hot path of a DFlash speculative-decoding draft layer, as
 * vllm.cpp's qwen3_dflash.cpp runs it per draft step:
 *   1. context keys: per-head RMSNorm (k_norm) then NeoX RoPE at the context positions,
 *      stored as bf16; V stored raw                 (PrecomputeContextKVDevice and
 *      AppendContextKVDevice, which scatter new rows into the context store);
 *   2. block q / k: per-head RMSNorm (q_norm / k_norm) then NeoX RoPE at the block
 *      positions                                     (ForwardWithCtxKVDev, ForwardPagedBody);
 *   3. block attention: every block row of request r attends to the request's context
 *      rows and to its own block rows -- bidirectionally on full-attention layers,
 *      causally with a sliding window on SWA layers -- with grouped-query heads;
 *      only block rows are produced                (DFlashBlockAttention over the combined
 *      [context ; block] sequence, blocks rows gathered by IndexSelect; the paged variant
 *      computes only block rows).
 *
 * Conventions for every entry point
 *   - Pointers to tensors and metadata are DEVICE pointers owned by the caller; the
 *     library never frees or retains them. Tensors are dense, row-major, contiguous.
 *   - bf16 tensors are passed as dflash_bf16 (the 16-bit pattern of a bfloat16).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *     and runs asynchronously: the calls allocate no memory and do not synchronise.
 *   - Every call returns DFLASH_OK (0) or a negative status; dflash_last_error() then
 *     holds a message (thread-local). Nothing is thrown or aborts across this boundary.
 *   - Errors found from host arguments are reported before anything is enqueued.
 *     Errors that only device metadata can reveal (bad offsets, a bounded device wait
 *     that ran out) are recorded in the workspace and read by dflash_check_error().
 *   - Only sm_103a (GB300) devices are supported; no CPU or other-GPU fallback exists.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#if defined(DFLASH_BUILD) && defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dflash_bf16;   /* bfloat16 bit pattern */
typedef void* dflash_stream_t;  /* cudaStream_t */

enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1,   /* a host argument is out of range or inconsistent   */
  DFLASH_ERR_UNSUPPORTED = -2,   /* valid, but outside what the kernels implement      */
  DFLASH_ERR_WORKSPACE = -3,     /* workspace missing, misaligned or too small          */
  DFLASH_ERR_CUDA = -4,          /* a CUDA runtime call failed (message has the reason) */
  DFLASH_ERR_DEVICE_TIMEOUT = -5,/* a bounded device-side wait ran out                  */
  DFLASH_ERR_DEVICE_METADATA = -6/* device metadata was inconsistent (rows skipped)     */
};

enum {
  DFLASH_OUT_BF16 = 0,           /* out is bf16 [total_q, Hq, Dh]                       */
  DFLASH_OUT_F32 = 1             /* out is f32; computed with split (hi+lo) bf16 operands */
};

enum {
  DFLASH_FLAG_FORCE_SPLIT = 1,   /* always split each request's keys over several CTAs  */
  DFLASH_FLAG_NO_SPLIT = 2       /* never split (one CTA per request x kv head x q tile)*/
};

/* Message describing the last failing call on this thread ("" after success). */
DFLASH_API const char* dflash_last_error(void);

/* Library ABI version: (major << 16) | minor. */
DFLASH_API int dflash_version(void);

/*
 * dflash_context_kv -- write rows into the draft model's context K/V store.
 * (qwen3_dflash.cpp, PrecomputeContextKVDevice: k_norm over head_dim, then RopeNeox at
 *  the context positions, V raw; AppendContextKVDevice: new rows go to store slots.)
 *
 *   k_raw    bf16 [n, Hkv, Dh]  projected keys of the new rows (before k_norm)
 *   v        bf16 [n, Hkv, Dh]  projected values of the new rows; may be NULL (no V write)
 *   ctx_pos  int32 [n]          absolute position of each new row (RoPE angle)
 *   k_norm_w bf16 [Dh]          k_norm weight
 *   slot     int32 [n] or NULL  destination row of each new row in the store; NULL means
 *                               row i goes to row i. Slots must be distinct and in
 *                               [0, capacity); a row whose slot is out of range is skipped
 *                               (checked on device, not reported).
 *   ctx_k    bf16 [capacity, Hkv, Dh] store K: out[slot[i]] = rope(rmsnorm(k_raw[i]))
 *   ctx_v    bf16 [capacity, Hkv, Dh] store V: out[slot[i]] = v[i] (ignored if v is NULL)
 *   eps, rope_theta             RMSNorm epsilon, RoPE base (inv_freq_i = theta^(-2i/Dh))
 *   Dh in {64, 128}; Hkv >= 1. k_raw may alias ctx_k (and v ctx_v) when slot is NULL.
 *   Math: f32 RMSNorm and rotation with an exactly reduced angle; one bf16 rounding.
 */
DFLASH_API int dflash_context_kv(const dflash_bf16* k_raw, const dflash_bf16* v, const int32_t* ctx_pos,
                      const dflash_bf16* k_norm_w, const int32_t* slot, int64_t n, int hkv, int dh,
                      float eps, float rope_theta, dflash_bf16* ctx_k, dflash_bf16* ctx_v,
                      int64_t capacity, dflash_stream_t stream);

/*
 * Bytes of device workspace dflash_block_attention needs on the current device for these
 * arguments (same meaning as there). Returns 0 and sets the error message if the
 * arguments are invalid. The workspace needs no initialisation.
 */
DFLASH_API size_t dflash_block_attention_workspace_size(int num_reqs, int64_t total_q, int hq, int hkv, int dh,
                                                        int64_t total_ctx, int max_ctx_len, int max_block_len,
                                                        int causal, int window, int out_dtype, int flags);

/*
 * Describes how dflash_block_attention would run with these arguments on the current
 * device: plan[0] = kernel launches per call (prologue, attention and, when a request's
 * keys may be split over several CTAs, the combine pass), plan[1] = key tiles (128 keys)
 * per split, plan[2] = upper bound of work units, plan[3] = attention CTAs, plan[4] =
 * workspace bytes / 256 (rounded up). Returns DFLASH_OK or an error status.
 */
DFLASH_API int dflash_block_attention_plan(int num_reqs, int64_t total_q, int hq, int hkv, int dh, int64_t total_ctx,
                                           int max_ctx_len, int max_block_len, int causal, int window, int out_dtype,
                                           int flags, int64_t plan[5]);

/*
 * dflash_block_attention -- attention of every block row over [context ; block] of its
 * request, with the q/k RMSNorm + NeoX RoPE prologue fused in.
 * (qwen3_dflash.cpp: ForwardWithCtxKVDev builds per request the combined sequence
 *  [context rows ; block rows] (cu_comb / ctx_dest / blk_idx) and calls
 *  DFlashBlockAttention with scale = 1/sqrt(head_dim), causal and sliding_window from the
 *  layer, keeping only block rows; ForwardPagedBody computes only block rows directly.)
 *
 *   q_raw      bf16 [total_q, Hq, Dh]   block queries before q_norm
 *   k_blk      bf16 [total_q, Hkv, Dh]  block keys before k_norm
 *   v_blk      bf16 [total_q, Hkv, Dh]  block values
 *   ctx_k      bf16 [total_ctx, Hkv, Dh] stored context keys (normed + rotated, e.g. by
 *                                       dflash_context_kv)
 *   ctx_v      bf16 [total_ctx, Hkv, Dh] stored context values
 *   query_start_loc int32 [num_reqs+1]  block rows of request r are qsl[r] .. qsl[r+1]-1;
 *                                       qsl[0] = 0, nondecreasing, qsl[num_reqs] = total_q
 *   ctx_start_loc   int32 [num_reqs+1]  context segment of request r starts at row
 *                                       ctx_start_loc[r]; its capacity is
 *                                       ctx_start_loc[r+1] - ctx_start_loc[r]
 *   ctx_lens        int32 [num_reqs]    live context rows of request r (<= capacity): the
 *                                       first ctx_lens[r] rows of the segment
 *   positions       int32 [total_q]     block-row positions (RoPE angle of q and k_blk)
 *   q_norm_w, k_norm_w bf16 [Dh]        q_norm / k_norm weights
 *   num_reqs, total_q, Hq, Hkv, Dh      sizes; Hq % Hkv == 0, Dh in {64, 128}, Hq/Hkv <= 64
 *   total_ctx                           rows of ctx_k / ctx_v
 *   max_ctx_len, max_block_len          host upper bounds of ctx_lens[r] and of the block
 *                                       length; they size the grid and the workspace only
 *   eps, rope_theta                     RMSNorm epsilon and RoPE base
 *   scale                               score scale; <= 0 means 1/sqrt(Dh)
 *   causal, window                      causal = 0: every key of the request is visible;
 *                                       causal = 1: key j visible to query i iff j <= i in the
 *                                       combined order, and, if window > 0, i - j < window.
 *                                       window > 0 requires causal = 1.
 *   out_dtype, out                      DFLASH_OUT_BF16 or DFLASH_OUT_F32; out [total_q, Hq, Dh]
 *   workspace, workspace_bytes          device scratch of at least
 *                                       dflash_block_attention_workspace_size(...) bytes,
 *                                       256-byte aligned; reused across calls on one stream
 *   flags                               DFLASH_FLAG_* bits
 * Requests with no block rows produce nothing; requests with no context attend to their
 * block only. Concurrent calls must not share a workspace.
 */
DFLASH_API int dflash_block_attention(const dflash_bf16* q_raw, const dflash_bf16* k_blk, const dflash_bf16* v_blk,
                           const dflash_bf16* ctx_k, const dflash_bf16* ctx_v,
                           const int32_t* query_start_loc, const int32_t* ctx_start_loc,
                           const int32_t* ctx_lens, const int32_t* positions,
                           const dflash_bf16* q_norm_w, const dflash_bf16* k_norm_w,
                           int num_reqs, int64_t total_q, int hq, int hkv, int dh, int64_t total_ctx,
                           int max_ctx_len, int max_block_len, float eps, float rope_theta, float scale,
                           int causal, int window, int out_dtype, void* out, void* workspace,
                           size_t workspace_bytes, int flags, dflash_stream_t stream);

/*
 * dflash_block_attention_paged -- dflash_block_attention with the context in page pools.
 * (qwen3_dflash.cpp: the paged path, ForwardPagedBody, reads each layer's context K/V from
 *  [max_pages, page_size, Hkv, Dh] pools through a per-request block table and the device
 *  seq_lens, and writes new rows into page slots.)
 *
 *   k_pool, v_pool  bf16 [num_pages, page_size, Hkv, Dh]  context keys (normed + rotated,
 *                   e.g. by dflash_context_kv with slot = page * page_size + offset) and values
 *   block_table     int32 [num_reqs, max_pages_per_req]   request r's context row j is row
 *                   j % page_size of page block_table[r * max_pages_per_req + j / page_size]
 *   num_pages, page_size, max_pages_per_req                page_size in {16, 32, 64, 128};
 *                   max_ctx_len <= max_pages_per_req * page_size
 *   ctx_lens        int32 [num_reqs]  live context rows of request r (<= max_pages_per_req *
 *                   page_size); only the pages that hold them are read
 * Every other argument is that of dflash_block_attention (there is no ctx_start_loc). The
 * workspace is sized by dflash_block_attention_workspace_size with total_ctx =
 * num_pages * page_size. A block-table entry outside [0, num_pages) is recorded in the
 * device error word (DFLASH_ERR_DEVICE_METADATA through dflash_check_error) and page 0 is
 * read in its place.
 */
DFLASH_API int dflash_block_attention_paged(const dflash_bf16* q_raw, const dflash_bf16* k_blk,
                                            const dflash_bf16* v_blk, const dflash_bf16* k_pool,
                                            const dflash_bf16* v_pool, const int32_t* block_table, int64_t num_pages,
                                            int page_size, int max_pages_per_req, const int32_t* query_start_loc,
                                            const int32_t* ctx_lens, const int32_t* positions,
                                            const dflash_bf16* q_norm_w, const dflash_bf16* k_norm_w, int num_reqs,
                                            int64_t total_q, int hq, int hkv, int dh, int max_ctx_len,
                                            int max_block_len, float eps, float rope_theta, float scale, int causal,
                                            int window, int out_dtype, void* out, void* workspace,
                                            size_t workspace_bytes, int flags, dflash_stream_t stream);

/*
 * dflash_block_attention_noalloc -- dflash_block_attention without a caller workspace.
 * The pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory themselves (a plugin host that owns every byte of device
 * memory, code running inside another allocator's callback, deployments with a static
 * memory plan where a run-time cudaMalloc is not allowed). Arguments are those of
 * dflash_block_attention minus the workspace; inputs and output are still the caller's.
 * The scratch is a 32 MiB array compiled into the library: every GPU that loads the
 * library holds it until the process exits. A call whose workspace would exceed 32 MiB
 * (dflash_block_attention_workspace_size) fails with DFLASH_ERR_WORKSPACE and does
 * nothing. The first call on a device looks up the array's device address with that
 * device current and caches it; make that first call before any stream capture. All
 * calls on a device share the array, so calls that overlap on the GPU (two streams at
 * once) race and must not be issued. dflash_check_error cannot read this scratch; errors
 * of the call itself are returned and described by dflash_last_error.
 */
DFLASH_API int dflash_block_attention_noalloc(const dflash_bf16* q_raw, const dflash_bf16* k_blk,
                                              const dflash_bf16* v_blk, const dflash_bf16* ctx_k,
                                              const dflash_bf16* ctx_v, const int32_t* query_start_loc,
                                              const int32_t* ctx_start_loc, const int32_t* ctx_lens,
                                              const int32_t* positions, const dflash_bf16* q_norm_w,
                                              const dflash_bf16* k_norm_w, int num_reqs, int64_t total_q, int hq,
                                              int hkv, int dh, int64_t total_ctx, int max_ctx_len, int max_block_len,
                                              float eps, float rope_theta, float scale, int causal, int window,
                                              int out_dtype, void* out, int flags, dflash_stream_t stream);

/*
 * Reads the device error word the last dflash_block_attention call on this workspace
 * left (waits for `stream`). Returns DFLASH_OK, DFLASH_ERR_DEVICE_TIMEOUT or
 * DFLASH_ERR_DEVICE_METADATA; the word is cleared by the next attention call.
 */
DFLASH_API int dflash_check_error(const void* workspace, dflash_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H_ */
