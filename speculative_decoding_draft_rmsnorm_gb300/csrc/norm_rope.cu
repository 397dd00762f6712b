// norm_rope.cu -- host helpers and the stand-alone launch of the fused per-head
// RMSNorm + NeoX RoPE kernel (used for the context K/V store write).
#include <cmath>

#include "norm_rope.cuh"

namespace dflash {

void make_rope_turns(int dh, double theta, RopeTurns* out) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < kMaxHeadDim / 2; ++i) {
    double g = 0.0;
    if (i < dh / 2) g = std::pow(theta, -2.0 * i / dh) / two_pi;
    const float hi = static_cast<float>(g);
    out->hi[i] = hi;
    out->lo[i] = static_cast<float>(g - static_cast<double>(hi));
  }
}

template <int DH>
__global__ void __launch_bounds__(256) norm_rope_kernel(const __grid_constant__ NormRopeJob job) {
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  norm_rope_rows<DH>(job, warp_id, n_warps);
}

cudaError_t launch_norm_rope(const NormRopeJob& job, int dh, int num_sms, cudaStream_t stream) {
  if (job.n_tok <= 0) return cudaSuccess;
  const int64_t warps_needed = job.n_tok * norm_rope_items_per_token(job, dh);
  int64_t blocks = (warps_needed + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 4;  // a few waves of 8-warp blocks per SM
  if (blocks > cap) blocks = cap;
  if (dh == 128) {
    norm_rope_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(job);
  } else {
    norm_rope_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(job);
  }
  return cudaGetLastError();
}

// Start locations of up to this many requests are staged in shared memory for the row search.
constexpr int kAppendSmemReqs = 1024;

template <int DH>
__global__ void __launch_bounds__(256) append_rows_kernel(const __grid_constant__ NormRopeJob job,
                                                          const __grid_constant__ AppendMap map) {
  __shared__ int32_t s_nsl[kAppendSmemReqs + 1];
  AppendMap m = map;
  if (map.num_reqs <= kAppendSmemReqs) {
    for (int i = threadIdx.x; i <= map.num_reqs; i += blockDim.x) s_nsl[i] = map.new_start_loc[i];
    __syncthreads();
    m.new_start_loc = s_nsl;
  }
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  norm_rope_rows<DH, true, true>(job, warp_id, n_warps, &m);
}

cudaError_t launch_append_rows(const NormRopeJob& job, const AppendMap& map, int dh, int num_sms,
                               cudaStream_t stream) {
  if (job.n_tok <= 0) return cudaSuccess;
  const int64_t warps_needed = job.n_tok * norm_rope_items_per_token(job, dh);
  int64_t blocks = (warps_needed + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 4;
  if (blocks > cap) blocks = cap;
  if (dh == 128) {
    append_rows_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(job, map);
  } else {
    append_rows_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(job, map);
  }
  return cudaGetLastError();
}

}  // namespace dflash
