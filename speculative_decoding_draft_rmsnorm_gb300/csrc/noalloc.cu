// noalloc.cu -- dflash_block_attention_noalloc: block attention whose scratch lives in a
// fixed-size array compiled into the library, for callers that cannot allocate device
// memory themselves.
//
// Who needs it: plugin hosts that own every byte of device memory and hand out no
// scratch, code that runs inside another allocator's callback, and deployments with a
// static memory plan in which a cudaMalloc (which may synchronise the device and can
// fail at run time) is not allowed on the serving path. They still pass their own
// inputs and output; only the workspace moves into the library.
//
// The scratch array below is a file-scope __device__ variable: every GPU on which the
// library is loaded holds kScratchBytes for it until the process exits. On the host its
// name is only a stand-in for the device address, so the address is fetched once per
// device with cudaGetSymbolAddress (with that device current) and cached; the first
// call on each device does this set-up, so make that first call before any stream
// capture. Every call shares the one array per device, which keeps the previous call's
// contents (the kernels initialise everything they read), so calls that overlap on the
// GPU -- two streams at once -- race and must not be issued.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/dflash.h"
#include "internal.h"

static constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per device

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

struct ScratchCache {
  std::mutex mu;
  void* ptr[kMaxDevices] = {};
};

ScratchCache& cache() {
  static ScratchCache c;
  return c;
}

}  // namespace

extern "C" {

DFLASH_API int dflash_block_attention_noalloc(
    const dflash_bf16* q_raw, const dflash_bf16* k_blk, const dflash_bf16* v_blk, const dflash_bf16* ctx_k,
    const dflash_bf16* ctx_v, const int32_t* query_start_loc, const int32_t* ctx_start_loc, const int32_t* ctx_lens,
    const int32_t* positions, const dflash_bf16* q_norm_w, const dflash_bf16* k_norm_w, int num_reqs, int64_t total_q,
    int hq, int hkv, int dh, int64_t total_ctx, int max_ctx_len, int max_block_len, float eps, float rope_theta,
    float scale, int causal, int window, int out_dtype, void* out, int flags, dflash_stream_t stream) {
  const size_t need = dflash_block_attention_workspace_size(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len,
                                                            max_block_len, causal, window, out_dtype, flags);
  if (need == 0) return DFLASH_ERR_INVALID_ARG;  // the size query has set the message
  char msg[256];
  if (need > kScratchBytes) {
    std::snprintf(msg, sizeof msg,
                  "this call needs %zu bytes of scratch but the built-in scratch holds %zu; use "
                  "dflash_block_attention with a caller workspace",
                  need, kScratchBytes);
    return dflash::report_error(DFLASH_ERR_WORKSPACE, msg);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    std::snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    return dflash::report_error(DFLASH_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) {
    std::snprintf(msg, sizeof msg, "device %d: the built-in scratch serves devices 0 to %d only", dev,
                  kMaxDevices - 1);
    return dflash::report_error(DFLASH_ERR_UNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(cache().mu);
    scratch = cache().ptr[dev];
    if (!scratch) {
      e = cudaGetSymbolAddress(&scratch, g_scratch);
      if (e != cudaSuccess || !scratch) {
        std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        return dflash::report_error(DFLASH_ERR_CUDA, msg);
      }
      cache().ptr[dev] = scratch;
    }
  }
  return dflash_block_attention(q_raw, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens,
                                positions, q_norm_w, k_norm_w, num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len,
                                max_block_len, eps, rope_theta, scale, causal, window, out_dtype, out, scratch,
                                kScratchBytes, flags, stream);
}

// The device error word of the last noalloc call on the current device lives in the built-in
// scratch, which the caller has no pointer to; this reads it exactly as dflash_check_error
// reads a caller's workspace (it waits for `stream`).
DFLASH_API int dflash_block_attention_noalloc_check_error(dflash_stream_t stream) {
  char msg[160];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    std::snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    return dflash::report_error(DFLASH_ERR_CUDA, msg);
  }
  void* scratch = nullptr;
  if (dev >= 0 && dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(cache().mu);
    scratch = cache().ptr[dev];
  }
  if (!scratch) {
    std::snprintf(msg, sizeof msg, "no dflash_block_attention_noalloc call has run on device %d", dev);
    return dflash::report_error(DFLASH_ERR_INVALID_ARG, msg);
  }
  return dflash_check_error(scratch, stream);
}

}  // extern "C"
