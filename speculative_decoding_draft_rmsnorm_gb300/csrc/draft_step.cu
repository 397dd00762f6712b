// draft_step.cu -- the two integer-side steps around the draft model's attention:
//
//   dflash_paged_append    new context rows into a paged K/V store, lengths bumped on the device
//                          (vllm.cpp qwen3_dflash.cpp, AppendContextKVDevice);
//   dflash_prepare_inputs  the draft step's positions, slots, token ids and sample map
//                          (qwen3_dflash.cpp, PrepareDflashInputs).
//
// Both read every length from device memory and allocate nothing, so a captured graph replays
// them as the batch changes. Neither synchronises.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>

#include "../../include/dflash.h"
#include "internal.h"
#include "norm_rope.cuh"
#include "ptx.cuh"

namespace dflash {
namespace {

int failf(int code, const char* fmt, ...) {
  char buf[400];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  return report_error(code, buf);
}

int current_sms(int* out) {
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return failf(DFLASH_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return failf(DFLASH_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a (GB300) only", dev,
                 major, minor);
  return DFLASH_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ paged append: lengths
// Runs after the row kernel (programmatic launch: it waits for that grid to finish before it
// reads or writes anything), so every row saw the old lengths. One block: the start
// locations are checked first, and the lengths move only if all of them are consistent; then
// every request whose whole append fits (the row kernel's own test) grows by its count, and
// one that does not fit keeps its length and is reported.
__global__ void __launch_bounds__(1024) append_lengths_kernel(AppendMap m, int64_t n_rows, uint32_t* err) {
  grid_dependency_wait();
  int bad = 0;
  for (int r = threadIdx.x; r <= m.num_reqs; r += blockDim.x) {
    const int32_t a = m.new_start_loc[r];
    if (r == 0 && a < 0) bad = 1;
    if (r == m.num_reqs && a > n_rows) bad = 1;
    if (r < m.num_reqs && m.new_start_loc[r + 1] < a) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && err) atomicOr(err, kErrMetadata);
    return;
  }
  int overflow = 0;
  int32_t* lens = const_cast<int32_t*>(m.seq_lens);
  for (int r = threadIdx.x; r < m.num_reqs; r += blockDim.x) {
    if (append_fits(m, r, 0, 1))
      lens[r] += m.new_start_loc[r + 1] - m.new_start_loc[r];
    else
      overflow = 1;
  }
  if (__syncthreads_or(overflow) && threadIdx.x == 0 && err) atomicOr(err, kErrMetadata);
}

// ------------------------------------------------------------------ input preparation
struct PrepareArgs {
  const int32_t* idx_mapping;
  const int32_t* tqsl;  // target_query_start_loc [N+1]
  const int32_t* num_rejected;
  const int32_t* num_sampled;
  const int32_t* last_sampled;
  const int32_t* next_prefill;
  const int64_t* target_positions;
  const int32_t* block_table;
  int stride, num_reqs, nqpr, nspec, block_size, max_num_reqs, max_num_tokens, pad_token, anchor;
  int64_t n_tgt, max_model_len;
  int32_t* input_ids;
  int64_t* query_positions;
  int32_t* query_start_loc;
  int32_t* seq_lens;
  int64_t* query_slot_mapping;
  int64_t* context_positions;
  int64_t* context_slot_mapping;
  int32_t* sample_indices;
  int64_t* sample_pos;
  int32_t* sample_idx_mapping;
  uint32_t* err;
};

struct ReqInfo {
  int state;
  int bonus;
  int64_t last_pos;  // position of the last accepted context token
  bool ok;
};

__device__ __forceinline__ ReqInfo req_info(const PrepareArgs& a, int r) {
  ReqInfo q{0, 0, 0, false};
  const int state = a.idx_mapping[r];
  const int64_t accepted_end = static_cast<int64_t>(a.tqsl[r + 1]) - a.num_rejected[r];
  if (state < 0 || state >= a.max_num_reqs || accepted_end < 1 || accepted_end > a.n_tgt) return q;
  q.state = state;
  q.last_pos = a.target_positions[accepted_end - 1];
  q.bonus = a.num_sampled[r] > 0 ? a.last_sampled[state] : a.next_prefill[state];
  q.ok = true;
  return q;
}

// slot of position p of request r: its page (the table's last page past the end) and offset
__device__ __forceinline__ bool slot_of(const PrepareArgs& a, int r, int64_t p, int64_t* slot) {
  if (p < 0) return false;
  int64_t page = p / a.block_size;
  if (page > a.stride - 1) page = a.stride - 1;
  *slot = static_cast<int64_t>(a.block_table[static_cast<int64_t>(r) * a.stride + page]) * a.block_size +
          p % a.block_size;
  return true;
}

// One thread per output entry, over four ranges laid end to end: context tokens, query rows
// (max_num_tokens), request rows (max_num_reqs + 1) and sample rows (max_num_reqs * nspec).
// Every entry of every output is written exactly once.
__global__ void __launch_bounds__(256) prepare_inputs_kernel(const __grid_constant__ PrepareArgs a) {
  const int64_t n_ctx = a.n_tgt, n_q = a.max_num_tokens, n_r = a.max_num_reqs + 1;
  const int64_t n_s = static_cast<int64_t>(a.max_num_reqs) * a.nspec;
  const int64_t total = n_ctx + n_q + n_r + n_s;
  const int n = a.num_reqs;
  const int first = a.anchor ? 0 : 1;  // first sampled query offset
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < n_ctx) {  // context token t: its position and slot
      const int64_t t = i;
      int lo = 0, hi = n + 1;  // first r with tqsl[r] > t
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a.tqsl[mid] <= t) lo = mid + 1; else hi = mid;
      }
      const int r = lo - 1;
      int64_t p = 0, slot = 0;
      if (r >= 0 && r < n) {
        p = a.target_positions[t];
        if (!slot_of(a, r, p, &slot)) bad = true;
      }
      a.context_positions[t] = p;
      a.context_slot_mapping[t] = slot;
      continue;
    }
    int64_t j = i - n_ctx;
    if (j < n_q) {  // query row j
      if (j < static_cast<int64_t>(n) * a.nqpr) {
        const int r = static_cast<int>(j / a.nqpr), k = static_cast<int>(j % a.nqpr);
        const ReqInfo q = req_info(a, r);
        int64_t p = 0, slot = 0;
        if (q.ok) {
          p = q.last_pos + 1 + k;
          if (!slot_of(a, r, p, &slot)) bad = true;
        } else {
          bad = true;
        }
        a.input_ids[j] = k == 0 ? q.bonus : a.pad_token;
        a.query_positions[j] = p < a.max_model_len - 1 ? p : a.max_model_len - 1;
        a.query_slot_mapping[j] = slot;
      } else {
        a.query_slot_mapping[j] = -1;  // padding slot
      }
      continue;
    }
    j -= n_q;
    if (j < n_r) {  // request row j: where its queries start, its draft length
      const int r = static_cast<int>(j);
      a.query_start_loc[r] = (r < n ? r : n) * a.nqpr;
      if (r < a.max_num_reqs) {
        int32_t len = 0;
        if (r < n) {
          const ReqInfo q = req_info(a, r);
          if (q.ok) len = static_cast<int32_t>(q.last_pos + 1 + a.nqpr); else bad = true;
          if (a.tqsl[r + 1] < a.tqsl[r]) bad = true;
        }
        a.seq_lens[r] = len;
      }
      if (r == 0 && (a.tqsl[0] < 0 || a.tqsl[n] > a.n_tgt)) bad = true;
      continue;
    }
    j -= n_r;  // sample row j
    int32_t idx = 0, map = -1;
    int64_t sp = 0;
    if (j < static_cast<int64_t>(n) * a.nspec) {
      const int r = static_cast<int>(j / a.nspec), k = static_cast<int>(j % a.nspec) + first;
      map = 0;
      if (k < a.nqpr) {
        const ReqInfo q = req_info(a, r);
        if (q.ok) {
          idx = r * a.nqpr + k;
          sp = q.last_pos + 1 + k + (a.anchor ? 1 : 0);
          map = q.state;
        } else {
          bad = true;
        }
      }
    }
    a.sample_indices[j] = idx;
    a.sample_pos[j] = sp;
    a.sample_idx_mapping[j] = map;
  }
  if (bad && a.err) atomicOr(a.err, kErrMetadata);
}

}  // namespace
}  // namespace dflash

extern "C" {

int dflash_paged_append(const dflash_bf16* k_raw, const dflash_bf16* v, const int32_t* new_start_loc,
                        int32_t* seq_lens, const int32_t* block_table, const dflash_bf16* k_norm_w, int num_reqs,
                        int64_t n, int hkv, int dh, int page_size, int max_pages_per_req, int64_t num_pages,
                        float eps, float rope_theta, dflash_bf16* k_pool, dflash_bf16* v_pool, int32_t* status,
                        dflash_stream_t stream) {
  using namespace dflash;
  if (dh != 64 && dh != 128) return failf(DFLASH_ERR_UNSUPPORTED, "head_dim %d: only 64 and 128 are implemented", dh);
  if (hkv <= 0) return failf(DFLASH_ERR_INVALID_ARG, "Hkv must be positive");
  if (num_reqs < 0 || n < 0 || num_pages < 0) return failf(DFLASH_ERR_INVALID_ARG, "negative size argument");
  if (page_size <= 0 || max_pages_per_req <= 0)
    return failf(DFLASH_ERR_INVALID_ARG, "page_size and max_pages_per_req must be positive");
  if (n > 0x7fffffff) return failf(DFLASH_ERR_UNSUPPORTED, "more than 2^31 - 1 new rows");
  if (!(eps >= 0.0f) || !(rope_theta > 0.0f)) return failf(DFLASH_ERR_INVALID_ARG, "eps must be >= 0 and theta > 0");
  if (num_reqs == 0) return report_error(DFLASH_OK, "");
  if (!new_start_loc || !seq_lens || !block_table) return failf(DFLASH_ERR_INVALID_ARG, "null metadata pointer");
  if (n > 0 && (!k_raw || !k_norm_w || !k_pool || (v && !v_pool)))
    return failf(DFLASH_ERR_INVALID_ARG, "null tensor pointer");
  if (n > 0 && (!aligned16(k_raw) || !aligned16(k_pool) || !aligned16(k_norm_w) ||
                (v && (!aligned16(v) || !aligned16(v_pool)))))
    return failf(DFLASH_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  int sms = 0;
  int rc = current_sms(&sms);
  if (rc != DFLASH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = reinterpret_cast<uint32_t*>(status);
  if (n > 0) {
    NormRopeJob job{};
    job.nparts = 1;
    job.part[0] = NormRopePart{k_raw, k_norm_w, k_pool, nullptr, v, v ? v_pool : nullptr, hkv};
    job.n_tok = n;
    job.eps = eps;
    job.err = err;
    make_rope_turns(dh, static_cast<double>(rope_theta), &job.turns);
    AppendMap map{new_start_loc, seq_lens, block_table, num_reqs, max_pages_per_req, page_size, num_pages};
    cudaError_t e = launch_append_rows(job, map, dh, sms, st);
    if (e != cudaSuccess) return failf(DFLASH_ERR_CUDA, "append rows launch: %s", cudaGetErrorString(e));
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(num_reqs >= 1024 ? 1024 : ((num_reqs + 32) / 32) * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  AppendMap map{new_start_loc, seq_lens, block_table, num_reqs, max_pages_per_req, page_size, num_pages};
  cudaError_t e = cudaLaunchKernelEx(&cfg, append_lengths_kernel, map, n, err);
  if (e != cudaSuccess) return failf(DFLASH_ERR_CUDA, "append lengths launch: %s", cudaGetErrorString(e));
  return report_error(DFLASH_OK, "");
}

int dflash_prepare_inputs(const int32_t* idx_mapping, const int32_t* target_query_start_loc,
                          const int32_t* num_rejected, const int32_t* num_sampled, const int32_t* last_sampled,
                          const int32_t* next_prefill_tokens, const int64_t* target_positions,
                          const int32_t* block_table, int block_table_stride, int num_reqs, int64_t num_target_tokens,
                          int num_query_per_req, int num_speculative_steps, int block_size, int max_num_reqs,
                          int max_num_tokens, int64_t max_model_len, int parallel_drafting_token_id,
                          int sample_from_anchor, int32_t* input_ids, int64_t* query_positions,
                          int32_t* query_start_loc, int32_t* seq_lens, int64_t* query_slot_mapping,
                          int64_t* context_positions, int64_t* context_slot_mapping, int32_t* sample_indices,
                          int64_t* sample_pos, int32_t* sample_idx_mapping, int32_t* status,
                          dflash_stream_t stream) {
  using namespace dflash;
  if (num_reqs <= 0) return failf(DFLASH_ERR_INVALID_ARG, "num_reqs must be positive");
  if (num_query_per_req <= 0 || num_speculative_steps < 0 || block_size <= 0 || block_table_stride <= 0 ||
      max_model_len <= 0 || num_target_tokens < 0)
    return failf(DFLASH_ERR_INVALID_ARG, "sizes must be positive (num_speculative_steps, num_target_tokens >= 0)");
  if (sample_from_anchor != 0 && sample_from_anchor != 1)
    return failf(DFLASH_ERR_INVALID_ARG, "sample_from_anchor must be 0 or 1");
  if (max_num_reqs < num_reqs) return failf(DFLASH_ERR_INVALID_ARG, "max_num_reqs < num_reqs");
  if (static_cast<int64_t>(num_reqs) * num_query_per_req > max_num_tokens)
    return failf(DFLASH_ERR_INVALID_ARG, "num_reqs * num_query_per_req exceeds max_num_tokens");
  if (num_query_per_req - (sample_from_anchor ? 0 : 1) > num_speculative_steps)
    return failf(DFLASH_ERR_INVALID_ARG, "%d sampled rows per request exceed num_speculative_steps=%d",
                 num_query_per_req - (sample_from_anchor ? 0 : 1), num_speculative_steps);
  if (static_cast<int64_t>(max_num_reqs) * num_speculative_steps > 0x7fffffff || num_target_tokens > 0x7fffffff)
    return failf(DFLASH_ERR_UNSUPPORTED, "output sizes must fit in int32");
  if (!idx_mapping || !target_query_start_loc || !num_rejected || !num_sampled || !last_sampled ||
      !next_prefill_tokens || (num_target_tokens > 0 && !target_positions) || !block_table || !input_ids ||
      !query_positions || !query_start_loc || !seq_lens || !query_slot_mapping ||
      (num_target_tokens > 0 && (!context_positions || !context_slot_mapping)) ||
      (num_speculative_steps > 0 && (!sample_indices || !sample_pos || !sample_idx_mapping)))
    return failf(DFLASH_ERR_INVALID_ARG, "null pointer");
  int sms = 0;
  int rc = current_sms(&sms);
  if (rc != DFLASH_OK) return rc;
  PrepareArgs a{};
  a.idx_mapping = idx_mapping;
  a.tqsl = target_query_start_loc;
  a.num_rejected = num_rejected;
  a.num_sampled = num_sampled;
  a.last_sampled = last_sampled;
  a.next_prefill = next_prefill_tokens;
  a.target_positions = target_positions;
  a.block_table = block_table;
  a.stride = block_table_stride;
  a.num_reqs = num_reqs;
  a.nqpr = num_query_per_req;
  a.nspec = num_speculative_steps;
  a.block_size = block_size;
  a.max_num_reqs = max_num_reqs;
  a.max_num_tokens = max_num_tokens;
  a.pad_token = parallel_drafting_token_id;
  a.anchor = sample_from_anchor;
  a.n_tgt = num_target_tokens;
  a.max_model_len = max_model_len;
  a.input_ids = input_ids;
  a.query_positions = query_positions;
  a.query_start_loc = query_start_loc;
  a.seq_lens = seq_lens;
  a.query_slot_mapping = query_slot_mapping;
  a.context_positions = context_positions;
  a.context_slot_mapping = context_slot_mapping;
  a.sample_indices = sample_indices;
  a.sample_pos = sample_pos;
  a.sample_idx_mapping = sample_idx_mapping;
  a.err = reinterpret_cast<uint32_t*>(status);
  const int64_t total = num_target_tokens + max_num_tokens + (max_num_reqs + 1) +
                        static_cast<int64_t>(max_num_reqs) * num_speculative_steps;
  int64_t blocks = (total + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
  prepare_inputs_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return failf(DFLASH_ERR_CUDA, "prepare inputs launch: %s", cudaGetErrorString(e));
  return report_error(DFLASH_OK, "");
}

}  // extern "C"
