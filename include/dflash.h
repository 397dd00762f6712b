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
 * Around it, two integer steps of the same draft step: the input preparation
 * (PrepareDflashInputs: positions, KV slots, token ids and the sample map) and the append
 * of new context rows to a paged store with the lengths advanced on the device
 * (AppendContextKVDevice).
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
 *     that ran out) are recorded in the workspace and read by dflash_check_error(), or,
 *     for the calls that take no workspace, ORed into a caller's device status word.
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

/* Bit that dflash_context_kv, dflash_paged_append and dflash_prepare_inputs OR into their
 * `status` word. */
enum { DFLASH_STATUS_METADATA = 2 /* a device index or length was out of range; see the call */ };

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
 *                               [0, capacity); a row whose slot is out of range is not
 *                               written (checked on device) and reported through status.
 *   ctx_k    bf16 [capacity, Hkv, Dh] store K: out[slot[i]] = rope(rmsnorm(k_raw[i]))
 *   ctx_v    bf16 [capacity, Hkv, Dh] store V: out[slot[i]] = v[i] (ignored if v is NULL)
 *   eps, rope_theta             RMSNorm epsilon, RoPE base (inv_freq_i = theta^(-2i/Dh))
 *   status   int32 device word or NULL: the call ORs DFLASH_STATUS_METADATA into it when a
 *                               row's slot is outside [0, capacity); it never clears it
 *   Dh in {64, 128}; Hkv >= 1. k_raw may alias ctx_k (and v ctx_v) when slot is NULL.
 *   Math: f32 RMSNorm and rotation with an exactly reduced angle; one bf16 rounding.
 */
DFLASH_API int dflash_context_kv(const dflash_bf16* k_raw, const dflash_bf16* v, const int32_t* ctx_pos,
                      const dflash_bf16* k_norm_w, const int32_t* slot, int64_t n, int hkv, int dh,
                      float eps, float rope_theta, dflash_bf16* ctx_k, dflash_bf16* ctx_v,
                      int64_t capacity, int32_t* status, dflash_stream_t stream);

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
 * once) race and must not be issued. Errors found from the host arguments are returned
 * and described by dflash_last_error; errors only the device can see (bad device metadata,
 * a bounded wait that ran out) are recorded in the built-in scratch and read with
 * dflash_block_attention_noalloc_check_error.
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
 * dflash_block_attention_noalloc_check_error -- dflash_check_error for the built-in scratch
 * of the current device: reads the device error word the last noalloc call on this device
 * left there (waits for `stream`). Returns DFLASH_OK, DFLASH_ERR_DEVICE_TIMEOUT or
 * DFLASH_ERR_DEVICE_METADATA; DFLASH_ERR_INVALID_ARG if no noalloc call has run on the
 * device. Allocates nothing.
 */
DFLASH_API int dflash_block_attention_noalloc_check_error(dflash_stream_t stream);

/*
 * dflash_paged_append -- append new context rows to a paged context K/V store and advance
 * each request's stored length on the device.
 * (qwen3_dflash.cpp, AppendContextKVDevice: the rows that follow a request's stored context
 *  take the positions [L, L + count), are projected as PrecomputeContextKVDevice does --
 *  k_norm over head_dim, then RopeNeox at that position, V raw -- and are scattered into
 *  the fixed page pools; the device seq_lens then becomes L + count, so a captured graph
 *  sees the longer context without a host copy.)
 *
 *   k_raw, v       bf16 [n, Hkv, Dh]  projected keys (before k_norm) and values of the new
 *                                     rows; v may be NULL (no V write)
 *   new_start_loc  int32 [N+1] device rows new_start_loc[r] .. new_start_loc[r+1] are request
 *                                     r's, in position order; rows outside
 *                                     [new_start_loc[0], new_start_loc[N]) are ignored
 *   seq_lens       int32 [N] device   in: stored length L_r; out: L_r + count_r. The same
 *                                     array dflash_block_attention_paged takes as ctx_lens
 *   block_table    int32 [N, max_pages_per_req] device, page ids of each request
 *   k_norm_w       bf16 [Dh]
 *   k_pool, v_pool bf16 [num_pages, page_size, Hkv, Dh]: new row i of request r (position
 *                                     p = L_r + i) goes to row p % page_size of page
 *                                     block_table[r, p / page_size]
 *   eps, rope_theta                   as dflash_context_kv (same kernel arithmetic)
 *   status         int32 device word or NULL. The call ORs DFLASH_STATUS_METADATA into it
 *                  when a request's append does not fit -- one of its new rows would fall
 *                  past its block table or on a page id outside the pool: like the page's
 *                  capacity check, which comes before any write, none of that request's
 *                  rows is written and its length stays; the other requests append -- or
 *                  when new_start_loc is not nondecreasing within [0, n] (then no length
 *                  moves). The call never clears it.
 *   Dh in {64, 128}; any page_size >= 1. Two launches: the rows, then the lengths (which
 *   waits for the rows, so every row sees the old length). Allocates nothing.
 */
DFLASH_API int dflash_paged_append(const dflash_bf16* k_raw, const dflash_bf16* v, const int32_t* new_start_loc,
                                   int32_t* seq_lens, const int32_t* block_table, const dflash_bf16* k_norm_w,
                                   int num_reqs, int64_t n, int hkv, int dh, int page_size, int max_pages_per_req,
                                   int64_t num_pages, float eps, float rope_theta, dflash_bf16* k_pool,
                                   dflash_bf16* v_pool, int32_t* status, dflash_stream_t stream);

/*
 * dflash_prepare_inputs -- the draft step's input preparation, as one integer kernel.
 * (qwen3_dflash.cpp, PrepareDflashInputs, the host form of vLLM's
 *  _prepare_dflash_inputs_kernel.) For every request r of the batch (state
 *  s = idx_mapping[r]; its target tokens target_query_start_loc[r] .. [r+1], of which the
 *  last num_rejected[r] were rejected; P = position of the last accepted one):
 *   context_positions[t] = target_positions[t], context_slot_mapping[t] = slot(r, that);
 *   query row r*Q + k (k < Q = num_query_per_req) at position P + 1 + k: input_ids = the
 *     bonus token (last_sampled[s] if num_sampled[r] > 0, else next_prefill_tokens[s]) for
 *     k = 0 and parallel_drafting_token_id after; query_positions = min(P + 1 + k,
 *     max_model_len - 1); query_slot_mapping = slot(r, P + 1 + k);
 *   query_start_loc[r] = r*Q; seq_lens[r] = P + 1 + Q;
 *   sample rows r*S + j (S = num_speculative_steps) for query offsets k = j + (0 when
 *     sample_from_anchor, else 1) < Q: sample_indices = r*Q + k, sample_pos = P + 1 + k
 *     (+1 when sample_from_anchor), sample_idx_mapping = s; later rows of the request 0.
 *  with slot(r, p) = block_table[r, min(p / block_size, stride - 1)] * block_size +
 *  p % block_size. Past the live requests: query_start_loc = N*Q, seq_lens 0, sample rows
 *  (0, 0, -1), query_slot_mapping -1; context entries past target_query_start_loc[N] are 0.
 *
 *   inputs (device): idx_mapping, num_rejected, num_sampled int32 [N];
 *     target_query_start_loc int32 [N+1]; last_sampled, next_prefill_tokens int32
 *     [max_num_reqs] (indexed by request state); target_positions int64
 *     [num_target_tokens]; block_table int32 [N, block_table_stride]
 *   outputs (device): input_ids int32 [N*Q]; query_positions int64 [N*Q]; query_start_loc
 *     int32 [max_num_reqs+1]; seq_lens int32 [max_num_reqs]; query_slot_mapping int64
 *     [max_num_tokens]; context_positions, context_slot_mapping int64 [num_target_tokens];
 *     sample_indices int32, sample_pos int64, sample_idx_mapping int32 [max_num_reqs*S]
 *   Requires N <= max_num_reqs, N*Q <= max_num_tokens and Q - (1 - sample_from_anchor) <= S
 *   (else DFLASH_ERR_INVALID_ARG). status: int32 device word or NULL; the call ORs
 *   DFLASH_STATUS_METADATA into it when a request state is outside [0, max_num_reqs), an
 *   accepted end falls outside the target tokens, a position is negative or
 *   target_query_start_loc is inconsistent (the affected entries are written as 0).
 *   One launch; allocates nothing; every output entry is written.
 */
DFLASH_API int dflash_prepare_inputs(const int32_t* idx_mapping, const int32_t* target_query_start_loc,
                                     const int32_t* num_rejected, const int32_t* num_sampled,
                                     const int32_t* last_sampled, const int32_t* next_prefill_tokens,
                                     const int64_t* target_positions, const int32_t* block_table,
                                     int block_table_stride, int num_reqs, int64_t num_target_tokens,
                                     int num_query_per_req, int num_speculative_steps, int block_size,
                                     int max_num_reqs, int max_num_tokens, int64_t max_model_len,
                                     int parallel_drafting_token_id, int sample_from_anchor, int32_t* input_ids,
                                     int64_t* query_positions, int32_t* query_start_loc, int32_t* seq_lens,
                                     int64_t* query_slot_mapping, int64_t* context_positions,
                                     int64_t* context_slot_mapping, int32_t* sample_indices, int64_t* sample_pos,
                                     int32_t* sample_idx_mapping, int32_t* status, dflash_stream_t stream);

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
