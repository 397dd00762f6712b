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

// Paged append: new row t belongs to request r when new_start_loc[r] <= t < new_start_loc[r+1];
// it takes position seq_lens[r] + (t - new_start_loc[r]) and lands at row position % page_size
// of page block_table[r, position / page_size] of the pool.
struct AppendMap {
  const int32_t* new_start_loc;  // [num_reqs + 1]
  const int32_t* seq_lens;       // [num_reqs], the lengths before this append
  const int32_t* block_table;    // [num_reqs, max_pages]
  int num_reqs, max_pages, page_size;
  int64_t num_pages;
};

// Norm + rope of the job's rows (pos and slot unused) into the rows the map gives.
cudaError_t launch_append_rows(const NormRopeJob& job, const AppendMap& map, int dh, int num_sms,
                               cudaStream_t stream);

// Work items (warp tasks) per token of a norm+rope job: heads are taken in chunks of
// 4 * 32 / (Dh / 8) per item.
inline int norm_rope_items_per_token(const NormRopeJob& job, int dh) {
  const int hpi = 4 * (32 / (dh / 8));
  int n = (job.part[0].heads + hpi - 1) / hpi;
  if (job.nparts > 1) n += (job.part[1].heads + hpi - 1) / hpi;
  return n;
}

// One group of the attention kernel's work: (request, kv head, query tile) with its n key
// tiles (context tiles first, then block tiles) at global tile indices [start, start+n).
struct Group {
  int r, kvh, qt, n;
  int start, clen, blen, ctx_lo;
  int n_ctx_tiles, csl, qsl, rows;  // rows of this query tile (G heads x tokens)
  int tok0, pad0, pad1, pad2;       // tok0 = first block index of the query tile
};
static_assert(sizeof(Group) == 64, "group descriptor is 64 bytes");

// Balanced schedule: what CTA c of the attention kernel needs before its first loads.
struct CtaRecord {
  Group first;         // the group holding the CTA's first tile
  int g0, lo, hi, ng;  // its index; the CTA's tiles [lo, hi); the number of groups
};
static_assert(sizeof(CtaRecord) == 80, "CTA record is 80 bytes");

struct AttnHost {
  // sizes
  int num_reqs, hq, hkv, dh, g, tpq, qt_max;
  int64_t total_q, total_ctx;
  int causal, window, out_f32, precise;
  float eps, scale_log2;
  int groups_max, grid;
  int max_ctx_len, max_block_len;
  bool balanced;
  int num_sms;
  // device pointers
  const uint16_t *q, *k_blk, *v_blk, *ctx_k, *ctx_v, *q_norm_w, *k_norm_w;
  const int32_t *qsl, *csl, *clen, *positions;  // csl: contiguous context only
  // paged context: ctx_k / ctx_v are pools of page_size-row pages; request r's context row j
  // is pool row block_table[r * max_pages + j / page_size] * page_size + j % page_size
  bool paged;
  const int32_t* block_table;
  int max_pages, page_size;
  void* out;
  // workspace carve-up
  uint32_t* ws_hdr;   // [0] error word, [1] group count, [2] total key tiles
  uint16_t *q_hat, *q_lo, *k_hat, *k_lo;
  Group* groups;
  CtaRecord* cta_rec; // [grid] balanced schedule only
  float* part_o;      // [2 * grid][64 * dh]  partial O of straddling segments (in thread order)
  float* part_ml;     // [2 * grid][64][2]   their running max (log2 units) and weight sum
  RopeTurns turns;
};

struct WorkspacePlan {
  size_t hdr, q_hat, q_lo, k_hat, k_lo, groups, cta_rec, part_o, part_ml, total;
  int groups_max, grid, parts, qt_max, tpq;
  double tiles_bound;
  bool balanced;
};

WorkspacePlan plan_workspace(int num_reqs, int64_t total_q, int hq, int hkv, int dh, int64_t total_ctx,
                             int max_ctx_len, int max_block_len, int window, int causal, int precise, int flags,
                             int num_sms);

cudaError_t launch_attention(const AttnHost& h, cudaStream_t stream, char* msg, size_t msg_len);

// Records `msg` as the thread's last error (what dflash_last_error returns) and returns code.
int report_error(int code, const char* msg);

}  // namespace dflash
