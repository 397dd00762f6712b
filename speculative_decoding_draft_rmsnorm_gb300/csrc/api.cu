// api.cu -- the extern "C" entry points declared in include/dflash.h: argument
// validation, workspace carve-up and kernel launches. No entry point allocates,
// synchronises (except dflash_check_error, which reads the device error word) or
// throws.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/dflash.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_msg[0] = '\0';
  return DFLASH_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sms(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *out = cache[dev];
    return DFLASH_OK;
  }
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return fail(DFLASH_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a (GB300) only", dev,
                major, minor);
  if (dev >= 0 && dev < 64) cache[dev] = sms;
  *out = sms;
  return DFLASH_OK;
}

int check_heads(int hq, int hkv, int dh) {
  if (dh != 64 && dh != 128) return fail(DFLASH_ERR_UNSUPPORTED, "head_dim %d: only 64 and 128 are implemented", dh);
  if (hkv <= 0 || hq <= 0) return fail(DFLASH_ERR_INVALID_ARG, "head counts must be positive (Hq=%d, Hkv=%d)", hq, hkv);
  if (hq % hkv) return fail(DFLASH_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", hq, hkv);
  if (hq / hkv > dflash::kTileRows)
    return fail(DFLASH_ERR_UNSUPPORTED, "group size Hq/Hkv=%d exceeds %d", hq / hkv, dflash::kTileRows);
  return DFLASH_OK;
}

int check_sizes(int num_reqs, int64_t total_q, int hq, int hkv, int dh, int64_t total_ctx, int max_ctx_len,
                int max_block_len, int out_dtype) {
  int rc = check_heads(hq, hkv, dh);
  if (rc != DFLASH_OK) return rc;
  if (num_reqs < 0 || total_q < 0 || total_ctx < 0 || max_ctx_len < 0 || max_block_len < 0)
    return fail(DFLASH_ERR_INVALID_ARG, "negative size argument");
  if (total_q > 0x7fffffff - 256 || total_ctx > 0x7fffffff - 256)
    return fail(DFLASH_ERR_UNSUPPORTED, "row counts must fit in int32 (total_q=%lld, total_ctx=%lld)",
                static_cast<long long>(total_q), static_cast<long long>(total_ctx));
  if (total_q > 0 && max_block_len == 0) return fail(DFLASH_ERR_INVALID_ARG, "max_block_len is 0 but total_q > 0");
  if (out_dtype != DFLASH_OUT_BF16 && out_dtype != DFLASH_OUT_F32)
    return fail(DFLASH_ERR_INVALID_ARG, "out_dtype %d is neither DFLASH_OUT_BF16 nor DFLASH_OUT_F32", out_dtype);
  return DFLASH_OK;
}

}  // namespace

namespace dflash {
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace dflash

extern "C" {

const char* dflash_last_error(void) { return g_msg; }

int dflash_version(void) { return (1 << 16) | 0; }

int dflash_context_kv(const dflash_bf16* k_raw, const dflash_bf16* v, const int32_t* ctx_pos,
                      const dflash_bf16* k_norm_w, const int32_t* slot, int64_t n, int hkv, int dh, float eps,
                      float rope_theta, dflash_bf16* ctx_k, dflash_bf16* ctx_v, int64_t capacity,
                      int32_t* status, dflash_stream_t stream) {
  if (dh != 64 && dh != 128) return fail(DFLASH_ERR_UNSUPPORTED, "head_dim %d: only 64 and 128 are implemented", dh);
  if (hkv <= 0) return fail(DFLASH_ERR_INVALID_ARG, "Hkv must be positive");
  if (n < 0 || capacity < 0) return fail(DFLASH_ERR_INVALID_ARG, "negative row count");
  if (!slot && n > capacity) return fail(DFLASH_ERR_INVALID_ARG, "n=%lld rows exceed capacity=%lld without slots",
                                         static_cast<long long>(n), static_cast<long long>(capacity));
  if (!(eps >= 0.0f) || !(rope_theta > 0.0f)) return fail(DFLASH_ERR_INVALID_ARG, "eps must be >= 0 and theta > 0");
  if (n == 0) return ok();
  if (!k_raw || !ctx_pos || !k_norm_w || !ctx_k || (v && !ctx_v))
    return fail(DFLASH_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(k_raw) || !aligned16(ctx_k) || !aligned16(k_norm_w) || (v && (!aligned16(v) || !aligned16(ctx_v))))
    return fail(DFLASH_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (slot && v && v == ctx_v) return fail(DFLASH_ERR_INVALID_ARG, "v may not alias ctx_v when slots are given");
  if (slot && k_raw == ctx_k) return fail(DFLASH_ERR_INVALID_ARG, "k_raw may not alias ctx_k when slots are given");
  int sms = 0;
  int rc = device_sms(&sms);
  if (rc != DFLASH_OK) return rc;
  dflash::NormRopeJob job{};
  job.nparts = 1;
  const bool copy_v = v != nullptr && v != ctx_v;
  job.part[0] = dflash::NormRopePart{k_raw, k_norm_w, ctx_k, nullptr, copy_v ? v : nullptr, copy_v ? ctx_v : nullptr,
                                     hkv};
  job.n_tok = n;
  job.pos = ctx_pos;
  job.slot = slot;
  job.capacity = capacity;
  job.eps = eps;
  job.err = reinterpret_cast<uint32_t*>(status);
  dflash::make_rope_turns(dh, static_cast<double>(rope_theta), &job.turns);
  cudaError_t e = dflash::launch_norm_rope(job, dh, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "norm_rope launch: %s", cudaGetErrorString(e));
  return ok();
}

size_t dflash_block_attention_workspace_size(int num_reqs, int64_t total_q, int hq, int hkv, int dh,
                                             int64_t total_ctx, int max_ctx_len, int max_block_len, int causal,
                                             int window, int out_dtype, int flags) {
  if (check_sizes(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len, out_dtype) != DFLASH_OK)
    return 0;
  if (causal != 0 && causal != 1) return fail(DFLASH_ERR_INVALID_ARG, "causal must be 0 or 1"), 0;
  if (window < 0 || (window > 0 && !causal)) return fail(DFLASH_ERR_INVALID_ARG, "window needs causal=1"), 0;
  int sms = 0;
  if (device_sms(&sms) != DFLASH_OK) return 0;
  const dflash::WorkspacePlan w = dflash::plan_workspace(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len,
                                                         max_block_len, window, causal, out_dtype == DFLASH_OUT_F32,
                                                         flags, sms);
  ok();
  return w.total;
}

int dflash_block_attention_plan(int num_reqs, int64_t total_q, int hq, int hkv, int dh, int64_t total_ctx,
                                int max_ctx_len, int max_block_len, int causal, int window, int out_dtype, int flags,
                                int64_t plan[5]) {
  int rc = check_sizes(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len, out_dtype);
  if (rc != DFLASH_OK) return rc;
  if (!plan) return fail(DFLASH_ERR_INVALID_ARG, "null plan array");
  if (causal != 0 && causal != 1) return fail(DFLASH_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window < 0 || (window > 0 && !causal)) return fail(DFLASH_ERR_INVALID_ARG, "window needs causal=1");
  int sms = 0;
  rc = device_sms(&sms);
  if (rc != DFLASH_OK) return rc;
  const dflash::WorkspacePlan w = dflash::plan_workspace(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len,
                                                         max_block_len, window, causal, out_dtype == DFLASH_OUT_F32,
                                                         flags, sms);
  const bool any = num_reqs > 0 && total_q > 0;
  plan[0] = any ? ((w.balanced && w.grid > 1) ? 3 : 2) : 0;  // the combine runs only with several CTAs
  plan[1] = static_cast<int64_t>(std::ceil(w.tiles_bound / w.grid));
  plan[2] = w.groups_max;
  plan[3] = any ? w.grid : 0;
  plan[4] = static_cast<int64_t>((w.total + 255) / 256);
  return ok();
}

}  // extern "C"

// Both attention entry points: contiguous context segments (block_table == nullptr) or
// paged pools (ctx_k / ctx_v are the pools, viewed as total_ctx = num_pages * page_size rows).
static int attention_call(const dflash_bf16* q_raw, const dflash_bf16* k_blk, const dflash_bf16* v_blk,
                          const dflash_bf16* ctx_k, const dflash_bf16* ctx_v, const int32_t* query_start_loc,
                          const int32_t* ctx_start_loc, const int32_t* ctx_lens, const int32_t* positions,
                          const dflash_bf16* q_norm_w, const dflash_bf16* k_norm_w, int num_reqs, int64_t total_q,
                          int hq, int hkv, int dh, int64_t total_ctx, int max_ctx_len, int max_block_len, float eps,
                          float rope_theta, float scale, int causal, int window, int out_dtype, void* out,
                          void* workspace, size_t workspace_bytes, int flags, dflash_stream_t stream, bool paged,
                          const int32_t* block_table, int max_pages, int page_size) {
  int rc = check_sizes(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len, out_dtype);
  if (rc != DFLASH_OK) return rc;
  if (causal != 0 && causal != 1) return fail(DFLASH_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window < 0) return fail(DFLASH_ERR_INVALID_ARG, "window must be >= 0");
  if (window > 0 && !causal) return fail(DFLASH_ERR_INVALID_ARG, "a sliding window requires causal=1");
  if (!(eps >= 0.0f) || !(rope_theta > 0.0f) || !std::isfinite(scale))
    return fail(DFLASH_ERR_INVALID_ARG, "eps must be >= 0, theta > 0 and scale finite");
  if ((flags & ~3) != 0 || flags == 3) return fail(DFLASH_ERR_INVALID_ARG, "unknown or contradictory flags %d", flags);
  if (num_reqs == 0 || total_q == 0) return ok();
  if (!q_raw || !k_blk || !v_blk || !query_start_loc || (paged ? !block_table : !ctx_start_loc) || !ctx_lens ||
      !positions || !q_norm_w || !k_norm_w || !out || !workspace)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  if (total_ctx > 0 && (!ctx_k || !ctx_v)) return fail(DFLASH_ERR_INVALID_ARG, "null context K/V with total_ctx > 0");
  if (!aligned16(q_raw) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(out) || !aligned16(q_norm_w) ||
      !aligned16(k_norm_w) || (total_ctx > 0 && (!aligned16(ctx_k) || !aligned16(ctx_v))))
    return fail(DFLASH_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DFLASH_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  int sms = 0;
  rc = device_sms(&sms);
  if (rc != DFLASH_OK) return rc;
  const int precise = out_dtype == DFLASH_OUT_F32 ? 1 : 0;
  const dflash::WorkspacePlan w = dflash::plan_workspace(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len,
                                                         max_block_len, window, causal, precise, flags, sms);
  if (w.tiles_bound > 2.0e9)
    return fail(DFLASH_ERR_UNSUPPORTED, "too many key tiles for one call (%.3g)", w.tiles_bound);
  if (workspace_bytes < w.total)
    return fail(DFLASH_ERR_WORKSPACE, "workspace has %zu bytes; %zu are needed", workspace_bytes, w.total);
  char* ws = static_cast<char*>(workspace);
  dflash::AttnHost h{};
  h.num_reqs = num_reqs;
  h.hq = hq;
  h.hkv = hkv;
  h.dh = dh;
  h.g = hq / hkv;
  h.tpq = w.tpq;
  h.qt_max = w.qt_max;
  h.total_q = total_q;
  h.total_ctx = total_ctx;
  h.causal = causal;
  h.window = window;
  h.out_f32 = out_dtype == DFLASH_OUT_F32;
  h.precise = precise;
  h.eps = eps;
  const float sc = scale > 0.0f ? scale : 1.0f / std::sqrt(static_cast<float>(dh));
  h.scale_log2 = sc * 1.4426950408889634f;
  h.groups_max = w.groups_max;
  h.grid = w.grid;
  h.max_ctx_len = max_ctx_len;
  h.max_block_len = max_block_len;
  h.balanced = w.balanced;
  h.num_sms = sms;
  h.q = q_raw;
  h.k_blk = k_blk;
  h.v_blk = v_blk;
  h.ctx_k = ctx_k;
  h.ctx_v = ctx_v;
  h.q_norm_w = q_norm_w;
  h.k_norm_w = k_norm_w;
  h.qsl = query_start_loc;
  h.csl = ctx_start_loc;
  h.clen = ctx_lens;
  h.positions = positions;
  h.paged = paged;
  h.block_table = block_table;
  h.max_pages = max_pages;
  h.page_size = page_size;
  h.out = out;
  h.ws_hdr = reinterpret_cast<uint32_t*>(ws + w.hdr);
  h.q_hat = reinterpret_cast<uint16_t*>(ws + w.q_hat);
  h.q_lo = precise ? reinterpret_cast<uint16_t*>(ws + w.q_lo) : nullptr;
  h.k_hat = reinterpret_cast<uint16_t*>(ws + w.k_hat);
  h.k_lo = precise ? reinterpret_cast<uint16_t*>(ws + w.k_lo) : nullptr;
  h.groups = reinterpret_cast<dflash::Group*>(ws + w.groups);
  h.cta_rec = w.balanced ? reinterpret_cast<dflash::CtaRecord*>(ws + w.cta_rec) : nullptr;
  h.part_o = w.balanced ? reinterpret_cast<float*>(ws + w.part_o) : nullptr;
  h.part_ml = w.balanced ? reinterpret_cast<float*>(ws + w.part_ml) : nullptr;
  dflash::make_rope_turns(dh, static_cast<double>(rope_theta), &h.turns);
  char msg[256] = "";
  cudaError_t e = dflash::launch_attention(h, static_cast<cudaStream_t>(stream), msg, sizeof msg);
  if (e != cudaSuccess)
    return fail(DFLASH_ERR_CUDA, "block attention launch: %s%s%s", cudaGetErrorString(e), msg[0] ? ": " : "", msg);
  return ok();
}

extern "C" {

int dflash_block_attention(const dflash_bf16* q_raw, const dflash_bf16* k_blk, const dflash_bf16* v_blk,
                           const dflash_bf16* ctx_k, const dflash_bf16* ctx_v, const int32_t* query_start_loc,
                           const int32_t* ctx_start_loc, const int32_t* ctx_lens, const int32_t* positions,
                           const dflash_bf16* q_norm_w, const dflash_bf16* k_norm_w, int num_reqs, int64_t total_q,
                           int hq, int hkv, int dh, int64_t total_ctx, int max_ctx_len, int max_block_len, float eps,
                           float rope_theta, float scale, int causal, int window, int out_dtype, void* out,
                           void* workspace, size_t workspace_bytes, int flags, dflash_stream_t stream) {
  return attention_call(q_raw, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens, positions,
                        q_norm_w, k_norm_w, num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len, eps,
                        rope_theta, scale, causal, window, out_dtype, out, workspace, workspace_bytes, flags, stream,
                        false, nullptr, 0, 0);
}

int dflash_block_attention_paged(const dflash_bf16* q_raw, const dflash_bf16* k_blk, const dflash_bf16* v_blk,
                                 const dflash_bf16* k_pool, const dflash_bf16* v_pool, const int32_t* block_table,
                                 int64_t num_pages, int page_size, int max_pages_per_req,
                                 const int32_t* query_start_loc, const int32_t* ctx_lens, const int32_t* positions,
                                 const dflash_bf16* q_norm_w, const dflash_bf16* k_norm_w, int num_reqs,
                                 int64_t total_q, int hq, int hkv, int dh, int max_ctx_len, int max_block_len,
                                 float eps, float rope_theta, float scale, int causal, int window, int out_dtype,
                                 void* out, void* workspace, size_t workspace_bytes, int flags,
                                 dflash_stream_t stream) {
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return fail(DFLASH_ERR_UNSUPPORTED, "page_size %d: only 16, 32, 64 and 128 are implemented", page_size);
  if (num_pages < 0 || max_pages_per_req < 0) return fail(DFLASH_ERR_INVALID_ARG, "negative page count");
  if (num_pages > (0x7fffffffLL - 256) / page_size)
    return fail(DFLASH_ERR_UNSUPPORTED, "the pools must hold fewer than 2^31 rows (num_pages=%lld)",
                static_cast<long long>(num_pages));
  if (static_cast<int64_t>(max_pages_per_req) * page_size < max_ctx_len)
    return fail(DFLASH_ERR_INVALID_ARG, "max_ctx_len %d exceeds max_pages_per_req x page_size", max_ctx_len);
  return attention_call(q_raw, k_blk, v_blk, k_pool, v_pool, query_start_loc, nullptr, ctx_lens, positions, q_norm_w,
                        k_norm_w, num_reqs, total_q, hq, hkv, dh, num_pages * page_size, max_ctx_len, max_block_len,
                        eps, rope_theta, scale, causal, window, out_dtype, out, workspace, workspace_bytes, flags,
                        stream, true, block_table, max_pages_per_req, page_size);
}

int dflash_check_error(const void* workspace, dflash_stream_t stream) {
  if (!workspace) return fail(DFLASH_ERR_INVALID_ARG, "null workspace");
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
  if (word & dflash::kErrTimeout) return fail(DFLASH_ERR_DEVICE_TIMEOUT, "a bounded device wait ran out (word %u)", word);
  if (word & dflash::kErrMetadata)
    return fail(DFLASH_ERR_DEVICE_METADATA, "device metadata inconsistent; affected requests skipped (word %u)", word);
  return ok();
}

}  // extern "C"
