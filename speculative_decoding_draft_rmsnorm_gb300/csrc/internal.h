// internal.h -- declarations shared by the library's translation units (not part of
// the public C ABI, which is include/dflash.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dflash {

constexpr int kMaxHeadDim = 128;
constexpr int kTileKeys = 128;   // keys per K/V tile of the attention kernel
constexpr int kTileRows = 64;    // query rows (group heads x block tokens) per MMA tile

// RoPE frequencies of one head size, as turns (revolutions) per position: the exact
// value inv_freq_i / (2 pi) split into a float head and a float tail.
struct RopeTurns {
  float hi[kMaxHeadDim / 2];
  float lo[kMaxHeadDim / 2];
};

void make_rope_turns(int dh, double theta, RopeTurns* out);

// One part of a norm+rope job: rows [n_tok, heads, dh] of `src` normed with `w`,
// rotated at the job's positions and written to dst_hi (and the bf16 remainder to
// dst_lo if non-null) at row slot[t] (or t).
struct NormRopePart {
  const uint16_t* src;
  const uint16_t* w;
  uint16_t* dst_hi;
  uint16_t* dst_lo;
  const uint16_t* v_src;  // optional raw rows copied to v_dst at the same row
  uint16_t* v_dst;
  int heads;
};

struct NormRopeJob {
  NormRopePart part[2];
  int nparts;
  int64_t n_tok;
  const int32_t* pos;
  const int32_t* slot;   // nullable
  int64_t capacity;      // rows of the destination (slot bound)
  float eps;
  uint32_t* err;         // nullable device error word
  RopeTurns turns;
};

cudaError_t launch_norm_rope(const NormRopeJob& job, int dh, int num_sms, cudaStream_t stream);

// Work unit of the attention kernel: one (request, kv head, query tile) and a
// contiguous range [t0, t1) of that request's key tiles (context tiles first, then
// block tiles).
struct Unit {
  int r, kvh, qt, t0;
  int t1, split, nsplit, first;     // first = unit index of split 0 of this group
  int clen, blen, ctx_lo, n_ctx_tiles;
  int csl, qsl, rows, tok0;         // rows of this q tile; tok0 = first block index
};
static_assert(sizeof(Unit) == 64, "unit descriptor is 64 bytes");

struct AttnHost {
  // sizes
  int num_reqs, hq, hkv, dh, g, tpq, qt_max;
  int64_t total_q, total_ctx;
  int causal, window, out_f32, precise;
  float eps, scale_log2;
  int tiles_per_split, max_splits, units_max;
  int max_ctx_len, max_block_len;
  bool may_split;
  int num_sms;
  // device pointers
  const uint16_t *q, *k_blk, *v_blk, *ctx_k, *ctx_v, *q_norm_w, *k_norm_w;
  const int32_t *qsl, *csl, *clen, *positions;
  void* out;
  // workspace carve-up
  uint32_t* ws_hdr;   // [0] error word, [1] unit count
  uint16_t *q_hat, *q_lo, *k_hat, *k_lo;
  Unit* units;
  float* part_o;      // [units_max][64][dh]
  float* part_ml;     // [units_max][64][2]
  RopeTurns turns;
};

struct WorkspacePlan {
  size_t hdr, q_hat, q_lo, k_hat, k_lo, units, part_o, part_ml, total;
  int tiles_per_split, max_splits, units_max, qt_max, tpq;
  bool may_split;
};

WorkspacePlan plan_workspace(int num_reqs, int64_t total_q, int hq, int hkv, int dh, int64_t total_ctx,
                             int max_ctx_len, int max_block_len, int window, int causal, int precise, int flags,
                             int num_sms);

cudaError_t launch_attention(const AttnHost& h, cudaStream_t stream, char* msg, size_t msg_len);

}  // namespace dflash
