// attention.cu -- DFlash draft block attention on sm_103a (tcgen05 + TMEM + TMA).
//
// What is computed (vllm.cpp qwen3_dflash.cpp, ForwardWithCtxKVDev / ForwardPagedBody):
// for request r with C context rows and B block rows, block row b (combined index
// i = C + b) and query head h (kv head h / G),
//     out[b, h] = sum_j softmax_j(scale * <q^_b,h , k^_j>) v_j
// over the request's keys j in combined order [context ; block]; bidirectional, or
// causal (j <= i) with an optional window (i - j < W).
//
// Three launches, chained with programmatic dependent launch:
//   A  prologue: q^ = rope(rmsnorm(q)), k^blk = rope(rmsnorm(k_blk)) into the workspace
//      (bf16; in precise mode also the bf16 remainders), and, in its first kTableBlocks
//      blocks, the table of groups (request, kv head, query tile) with their key-tile
//      counts and prefix offsets, and one schedule record per attention CTA.
//   B  attention: persistent CTAs, one per SM. Balanced (stream-K) schedule: the groups'
//      key tiles are laid end to end and each CTA takes a contiguous range of equal cost
//      (a tile, plus a little more for every group it starts; balanced_first_tile), so
//      every CTA streams about the same work whatever the raggedness; a group that
//      straddles CTAs is processed as segments whose partials are combined in C.
//      Warp 0 streams Q / K / V tiles with TMA (128-byte swizzle); warp 1 issues
//      tcgen05 MMAs: S = Q K^T into tensor memory (M = 64 query rows = G heads x block
//      tokens, N = 128 keys), and O += P V (N = Dh) from P in shared memory; warps 2-5
//      run the online softmax (f32, base 2, lazy rescale of O in TMEM when the running
//      maximum grows by more than 2^8) and the epilogue. A segment covering a whole
//      group writes the normalised output; a partial segment writes (O, m, l) to one of
//      its CTA's two partial slots (first segment: 2c, last: 2c+1).
//   C  combine: merges the partials of each group that straddles CTAs:
//      o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
//
// TMEM map (512 columns): S[0] at column 0, S[1] at 128, O of even segments at 256 and of
// odd segments at 256 + Dh (a segment's first PV waits only for the epilogue two segments
// back). An M = 64 MMA puts query row rho in lane 32*(rho/16) + rho%16; softmax warp w
// (sub-partition w%4) owns rows 16*(w%4) .. +15, lanes 0-15 of the warp taking key columns
// 0-63 and lanes 16-31 columns 64-127 (tcgen05.ld 16x32bx2).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "norm_rope.cuh"
#include "ptx.cuh"

namespace dflash {

// ================================================================ kernel A
struct PrologueParams {
  NormRopeJob job;
  const int32_t *qsl, *csl, *clen;
  Group* groups;
  CtaRecord* cta_rec;  // balanced schedule: one record per CTA of kernel B (else null)
  int grid_b;          // CTAs of kernel B
  uint32_t* hdr;
  int64_t total_q, total_ctx;
  int num_reqs, hkv, g, tpq, causal, window;
  int groups_max, max_ctx_len, max_block_len;
  int blk_tile;  // keys per block-key tile: 128, or 64 when hi and lo halves share a tile
  int paged;     // paged context: no ctx_start_loc; capacity paged_cap rows per request
  int page_size, paged_cap;
};

__device__ __forceinline__ void load_group(const Group* groups, int g, Group& G) {
  const int4* src = reinterpret_cast<const int4*>(groups + g);
  int4* dst = reinterpret_cast<int4*>(&G);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = src[i];
}

struct ReqTiles {  // one request's share of the group table
  int r, cnt, QT, n, C, B, lo, nct, c0, q0, goff;
  long long toff;
};

__device__ __forceinline__ Group make_group(const ReqTiles& q, int k, int tpq, int g) {
  Group G;
  G.r = q.r;
  G.kvh = k / q.QT;
  G.qt = k % q.QT;
  G.n = q.n;
  G.start = static_cast<int>(q.toff + static_cast<long long>(k) * q.n);
  G.clen = q.C;
  G.blen = q.B;
  G.ctx_lo = q.lo;
  G.n_ctx_tiles = q.nct;
  G.csl = q.c0;
  G.qsl = q.q0;
  G.tok0 = G.qt * tpq;
  G.rows = min(tpq, q.B - G.tok0) * g;
  G.pad0 = G.pad1 = G.pad2 = 0;
  return G;
}

// a / b for 0 <= a, 0 < b: 32-bit division when both fit
__device__ __forceinline__ long long div_nonneg(long long a, long long b) {
  if (a <= 0xffffffffll && b <= 0xffffffffll) return static_cast<unsigned>(a) / static_cast<unsigned>(b);
  return a / b;
}

// floor(c * T / grid) for 0 <= c <= grid, T < 2^31: 32-bit division when the product fits
__device__ __forceinline__ long long cta_first_tile(long long c, long long T, long long grid) {
  const unsigned long long prod = static_cast<unsigned long long>(c) * static_cast<unsigned long long>(T);
  if (prod <= 0xffffffffull) return static_cast<unsigned>(prod) / static_cast<unsigned>(grid);
  return static_cast<long long>(prod / static_cast<unsigned long long>(grid));
}

// Cost of key tiles and of segment starts in the balanced schedule, in eighths of a tile: a
// CTA's time grows by about 1.25 tiles for every group it starts (the group's Q tile, the
// previous segment's epilogue), measured per CTA on the Qwen3-4B-shaped layers.
constexpr long long kTileCost = 8, kSegCost = 10;
static_assert(kTileCost == 8, "balanced_first_tile divides by kTileCost with a shift");

// First tile of CTA c (0 <= c <= grid) of the balanced schedule over T tiles in G groups
// (req: the requests' tile and group offsets, n_req of them). With at least 4 tiles a CTA
// the split balances tiles and segment starts: tile t of group gi starts at cost
// u_t = 8 t + 10 (gi + 1), and CTA c takes the tiles with u_t in [c W / grid, (c+1) W / grid),
// W = 8 T + 10 G. Consecutive tile starts are at most 18 apart and every interval spans at
// least 31, so no CTA is empty. With fewer tiles: an even split, and with fewer tiles than
// CTAs one tile to each of the first T CTAs; empty CTAs only ever follow the last tile.
__device__ long long balanced_first_tile(long long c, long long T, long long G, long long grid, const ReqTiles* req,
                                         int n_req) {
  if (c >= grid) return T;
  if (T < 4 * grid) return T >= grid ? cta_first_tile(c, T, grid) : (c < T ? c : T);
  const long long W = kTileCost * T + kSegCost * G;
  const long long w = div_nonneg(c * W, grid);
  auto ufirst = [&](int r) { return kTileCost * req[r].toff + kSegCost * (static_cast<long long>(req[r].goff) + 1); };
  if (ufirst(0) > w) return 0;
  int a = 0, z = n_req - 1;  // the last request whose first tile starts at or below w
  while (a < z) {
    const int m = (a + z + 1) >> 1;
    if (ufirst(m) <= w) a = m; else z = m - 1;
  }
  const ReqTiles& q = req[a];
  if (q.cnt == 0) return q.toff;
  const long long per = kTileCost * q.n + kSegCost;  // one group: its start and its tiles
  const long long d = w - ufirst(a);
  const long long k = div_nonneg(d, per);
  if (k >= q.cnt) return q.toff + static_cast<long long>(q.cnt) * q.n;
  const long long rem = d - k * per;
  long long j = (rem + kTileCost - 1) >> 3;  // tiles of group k that start below w (kTileCost = 8)
  if (j > q.n) j = q.n;
  return q.toff + k * q.n + j;
}

// Validates the device metadata and writes one Group per (request, kv head, query tile)
// with its key-tile count and the global index of its first tile (prefix over groups).
// hdr[1] = number of groups, hdr[2] = total tiles. For the balanced schedule it also
// writes each CTA's record: CTA c owns tiles [lo_c, lo_{c+1}) (balanced_first_tile; with
// more than 256 requests an even split, lo_c = c*T/grid), its first group is the one
// holding tile lo_c, and the record carries that group so that the CTA's first loads
// depend on one read.
//
// Blocks of 256 threads, `nparts` of them (even). Requests are taken 256 at a time: a thread
// loads its request's metadata (one round trip), the block scans the group and tile counts,
// then every thread writes groups of the chunk (its request found by a search over the scan
// in shared memory) and, with one chunk, one thread per CTA writes the CTA's record, so no
// thread walks a request's groups serially. With one chunk (at most 256 requests) each of
// the nparts blocks repeats the loads and the scan; the first half of them write equal
// shares of the groups, the second half equal shares of the records: the stores of the
// table, not its arithmetic, set the time of this step (the L2 is full of dirty lines from
// the previous work), so spreading them over several SMs shortens it. Only part 0 writes
// the header words; with several chunks part 0 does all the work.
__device__ void build_groups(const PrologueParams& p, int part, int nparts) {
  __shared__ ReqTiles s_req[256];
  __shared__ int s_cnt[256];  // inclusive scan of the chunk's group counts
  __shared__ int s_wg[8];
  __shared__ long long s_wt[8];
  __shared__ int s_bad_global;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool one_chunk = p.num_reqs <= 256;
  if (!one_chunk && part != 0) return;
  const bool lead = part == 0;  // writes the header words (error word, counts)
  if (tid == 0) {
    if (lead) p.hdr[0] = 0;  // error word of this call (only this block writes it before kernel B)
    s_bad_global = 0;
  }
  __syncthreads();
  const long long grid = p.grid_b;
  int run_g = 0;
  long long run_t = 0;
  for (int base = 0; base < p.num_reqs; base += 256) {
    ReqTiles q{};
    q.r = base + tid;
    if (q.r < p.num_reqs) {
      // all loads of the request are independent: one round trip
      q.q0 = p.qsl[q.r];
      const int q1 = p.qsl[q.r + 1];
      q.c0 = p.paged ? 0 : p.csl[q.r];
      const int c1 = p.paged ? p.paged_cap : p.csl[q.r + 1];
      q.C = p.clen[q.r];
      q.B = q1 - q.q0;
      if ((q.r == 0 && q.q0 != 0) || (q.r == p.num_reqs - 1 && q1 != p.total_q)) s_bad_global = 1;
      // paged: the request's capacity is its block table (page ids are checked where they are
      // read); contiguous: its segment must lie inside the store
      const bool seg_ok = p.paged ? true : (q.c0 >= 0 && c1 >= q.c0 && c1 <= p.total_ctx);
      const bool ok = q.B >= 0 && q.q0 >= 0 && q1 <= p.total_q && seg_ok && q.C >= 0 && q.C <= c1 - q.c0 &&
                      q.C <= p.max_ctx_len && q.B <= p.max_block_len;
      if (!ok) {
        if (lead) atomicOr(&p.hdr[0], kErrMetadata);
        q.B = 0;
      }
      if (q.B > 0) {
        q.lo = (p.causal && p.window > 0) ? max(0, q.C - p.window + 1) : 0;
        // paged: context tiles start on a page boundary (keys before the window are masked)
        if (p.paged) q.lo -= q.lo % p.page_size;
        q.nct = (q.C - q.lo + kTileKeys - 1) / kTileKeys;
        q.n = q.nct + (q.B + p.blk_tile - 1) / p.blk_tile;
        q.QT = (q.B + p.tpq - 1) / p.tpq;
        q.cnt = p.hkv * q.QT;
      }
    }
    // block-wide inclusive scans of the group and tile counts: warp shuffles, then warp totals
    int ic = q.cnt;
    long long it = static_cast<long long>(q.cnt) * q.n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int vc = __shfl_up_sync(0xffffffffu, ic, off);
      const long long vt = __shfl_up_sync(0xffffffffu, it, off);
      if (lane >= off) {
        ic += vc;
        it += vt;
      }
    }
    if (lane == 31) {
      s_wg[wid] = ic;
      s_wt[wid] = it;
    }
    __syncthreads();
    int wg_before = 0, chunk_g = 0;
    long long wt_before = 0, chunk_t = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      if (w < wid) {
        wg_before += s_wg[w];
        wt_before += s_wt[w];
      }
      chunk_g += s_wg[w];
      chunk_t += s_wt[w];
    }
    ic += wg_before;
    it += wt_before;
    q.goff = run_g + ic - q.cnt;
    q.toff = run_t + it - static_cast<long long>(q.cnt) * q.n;
    s_cnt[tid] = ic;
    s_req[tid] = q;
    __syncthreads();
    const bool fits = run_g + chunk_g <= p.groups_max && run_t + chunk_t <= 0x7fffffffLL;
    if (!fits && tid == 0 && lead) atomicOr(&p.hdr[0], kErrMetadata);
    // this part's share: with one chunk the first half of the parts write the groups and the
    // second half the CTA records, each a contiguous share; otherwise part 0 writes all
    const int half = nparts / 2;
    const int gshare = one_chunk ? (chunk_g + half - 1) / half : chunk_g;
    const int g_begin = one_chunk ? (part < half ? min(chunk_g, part * gshare) : chunk_g) : 0;
    const int g_end = one_chunk ? min(chunk_g, g_begin + gshare) : chunk_g;
    const int cshare = static_cast<int>((grid + half - 1) / half);
    const int c_begin = one_chunk ? (part >= half ? min(static_cast<int>(grid), (part - half) * cshare)
                                                  : static_cast<int>(grid))
                                  : 0;
    const int c_end = one_chunk ? min(static_cast<int>(grid), c_begin + cshare) : static_cast<int>(grid);
    for (int j = g_begin + tid; fits && j < g_end; j += blockDim.x) {
      int a = 0, b = 255;  // first request of the chunk whose inclusive count exceeds j
      while (a < b) {
        const int m = (a + b) >> 1;
        if (s_cnt[m] > j) b = m; else a = m + 1;
      }
      const ReqTiles& rq = s_req[a];
      const int gi = run_g + j;
      p.groups[gi] = make_group(rq, gi - rq.goff, p.tpq, p.g);
    }
    if (one_chunk && fits && p.cta_rec != nullptr && chunk_t > 0) {
      // one thread per CTA: its range, the request holding its first tile (the last request
      // whose first tile is <= lo: that one has groups), and the group within it
      for (int c = c_begin + tid; c < c_end; c += blockDim.x) {
        const long long lo = balanced_first_tile(c, chunk_t, chunk_g, grid, s_req, p.num_reqs);
        const long long hi = balanced_first_tile(c + 1, chunk_t, chunk_g, grid, s_req, p.num_reqs);
        int a = 0, z = p.num_reqs - 1;
        while (a < z) {
          const int m = (a + z + 1) >> 1;
          if (s_req[m].toff <= lo) a = m; else z = m - 1;
        }
        const ReqTiles& rq = s_req[a];
        const int k =
            rq.n > 0 ? static_cast<int>(static_cast<unsigned>(lo - rq.toff) / static_cast<unsigned>(rq.n)) : 0;
        CtaRecord rec;
        rec.first = make_group(rq, k, p.tpq, p.g);
        rec.g0 = rq.goff + k;
        rec.lo = static_cast<int>(lo);
        rec.hi = static_cast<int>(hi);
        rec.ng = chunk_g;
        p.cta_rec[c] = rec;
      }
    }
    run_g += chunk_g;
    run_t += chunk_t;
    __syncthreads();  // s_req and s_cnt are rewritten by the next chunk
  }
  if (s_bad_global || run_g > p.groups_max || run_t > 0x7fffffffLL) {
    // no work for kernel B (the last two cannot happen with valid host bounds)
    if (tid == 0 && lead) atomicOr(&p.hdr[0], kErrMetadata);
    run_g = 0;
    run_t = 0;
  }
  if (tid == 0 && lead) {
    p.hdr[1] = static_cast<uint32_t>(run_g);
    p.hdr[2] = static_cast<uint32_t>(run_t);
  }
  if (p.cta_rec == nullptr) return;
  if (run_t == 0) {
    // records written above (if any) are replaced: no CTA has work. Each part clears the
    // records it wrote (with several chunks part 0 is the only part and owns all of them).
    const int half = nparts / 2;
    const long long share = (grid + half - 1) / half;
    const long long lo_c = part >= half ? static_cast<long long>(part - half) * share : grid;
    const int c0 = one_chunk ? static_cast<int>(lo_c < grid ? lo_c : grid) : 0;
    const int c1 = one_chunk ? static_cast<int>(c0 + share < grid ? c0 + share : grid) : static_cast<int>(grid);
    for (int c = c0 + tid; c < c1; c += blockDim.x) p.cta_rec[c] = CtaRecord{};
    return;
  }
  if (!one_chunk) {
    // several chunks: the total is known only now; read the table back (this block wrote
    // it, and the barrier at the end of the last chunk made it visible to all its threads)
    for (int gi = tid; gi < run_g; gi += blockDim.x) {
      Group G;
      load_group(p.groups, gi, G);
      const long long st = G.start;
      // the CTAs whose first tile lies in [st, st + n): ceil(st*grid/T) .. ceil((st+n)*grid/T) - 1
      const long long c0 = (st * grid + run_t - 1) / run_t;
      long long c1 = ((st + G.n) * grid + run_t - 1) / run_t - 1;
      if (c1 > grid - 1) c1 = grid - 1;
      for (long long c = c0; c <= c1; ++c) {
        CtaRecord rec;
        rec.first = G;
        rec.g0 = gi;
        rec.lo = static_cast<int>(cta_first_tile(c, run_t, grid));
        rec.hi = static_cast<int>(cta_first_tile(c + 1, run_t, grid));
        rec.ng = run_g;
        p.cta_rec[c] = rec;
      }
    }
  }
}

// Blocks 0 .. kTableBlocks-1 build the group table and the CTA records; the others run the
// q / block-k norm + RoPE. Three blocks per SM (at most 85 registers a thread), so that the
// launch below, sized to one item per warp where it can be, is resident at once.
constexpr int kTableBlocks = 8;
static_assert(kTableBlocks % 2 == 0, "half the table blocks write groups, half write records");

template <int DH>
__global__ void __launch_bounds__(256, 3) prologue_kernel(const __grid_constant__ PrologueParams p) {
  grid_dependents_launch();
  if (blockIdx.x < kTableBlocks) {
    build_groups(p, static_cast<int>(blockIdx.x), kTableBlocks);
    return;
  }
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x - kTableBlocks) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x - kTableBlocks) * blockDim.x) >> 5;
  norm_rope_rows<DH, false>(p.job, warp_id, n_warps);
}

// ================================================================ kernel B
// With two Q buffers (bf16 output), a whole group's normalised rows go out through the
// segment's own Q buffer: each thread holds 64 columns of one row, which written straight to
// global memory scatters every 16-byte store over 32 rows; staged, each half-warp writes a full
// row. The buffer is free once the segment's O_FULL has landed (its last QK completed), and the
// producer reloads it (two segments later) only after the softmax warps have arrived on Q_EMPTY.
// With one Q buffer the next segment's Q would wait on this epilogue, which itself waits for the
// next segment's first tile, so that configuration stores directly.
template <int NQ, bool PRECISE>
constexpr bool kStagedOut = NQ >= 2 && !PRECISE;
// A partial slot (64 rows x DH f32) is stored in the order the softmax threads hold it: the
// thread of TMEM sub-partition sp and lane L (row 16 sp + L % 16, columns from (L / 16) DH / 2)
// writes its k-th 4-float group (columns + 4k .. 4k + 3) at float4 index
// (sp DH / 8 + k) 32 + L, so that each warp store covers 512 contiguous bytes.
template <int DH>
__device__ __forceinline__ int64_t part_o_index(int sp, int k, int lane) {
  return (static_cast<int64_t>(sp) * (DH / 8) + k) * 32 + lane;
}

// A K or V tile normally sits in shared memory as DH / 64 column blocks of 128 rows x 128
// bytes (128-byte swizzle), one TMA box per column block (and page). With 16-row pages and
// Dh = 128 that is 32 boxes of 2 KB per K + V tile, and the per-box cost of the TMA unit, not
// HBM, sets the rate. Paged context tiles with Dh = 128 are instead stored group-major: rows
// 8i .. 8i + 7 at i * kGroupBytes, column block nb at + nb * 1 KB, so that one box brings a
// whole page (16 boxes a tile, whatever the page size). The 8-row groups are still evenly
// spaced, now kGroupBytes apart, which is all the MMA descriptors need: S = Q K^T still takes
// the 128 keys in one MMA per 16 columns and PV 16 keys per MMA.
constexpr uint32_t kGroupBytes = 2048;  // one 8-row group of both 64-column blocks

// Shared-memory plan. NQ query buffers (hi, and lo in precise mode), two P buffers (hi,
// and lo in precise mode), an NK-stage K ring and an NV-stage V ring; 1024-byte aligned
// tiles (128-byte swizzle atoms).
template <int DH, int NK, int NV, int NQ, bool PRECISE>
struct Layout {
  static constexpr int NB = DH / 64;                  // 128-byte column blocks per row
  static constexpr int QB = kTileRows * DH * 2;       // Q tile (one part)
  static constexpr int QBT = QB * (PRECISE ? 2 : 1);  // one Q buffer: hi [+ lo]
  static constexpr int PB = kTileRows * kTileKeys * 2;  // P tile (one part)
  static constexpr int PBT = PB * (PRECISE ? 2 : 1);  // one P buffer: hi [+ lo]
  static constexpr int KB = kTileKeys * DH * 2;       // K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_P = OFF_Q + NQ * QBT;
  static constexpr int OFF_K = OFF_P + 2 * PBT;
  static constexpr int OFF_V = OFF_K + NK * KB;
  static constexpr int OFF_BAR = OFF_V + NV * KB;
  // barrier indices
  static constexpr int K_FULL = 0, K_EMPTY = NK, V_FULL = 2 * NK, V_EMPTY = 2 * NK + NV;
  static constexpr int Q_FULL = 2 * NK + 2 * NV, Q_EMPTY = Q_FULL + 2, S_FULL = Q_FULL + 4, S_EMPTY = Q_FULL + 6;
  static constexpr int P_FULL = Q_FULL + 8, P_EMPTY = Q_FULL + 10, O_FULL = Q_FULL + 12, O_EMPTY = Q_FULL + 14;
  static constexpr int DRAIN = Q_FULL + 16;  // final commit of the MMA thread (its own barrier)
  static constexpr int NBARS = Q_FULL + 17;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int OFF_REC = (OFF_MISC + 64 + 15) / 16 * 16;  // CtaRecord (80 bytes)
  static constexpr int BYTES = OFF_REC + 80;
  static constexpr int ALLOC = BYTES + 1024;
};

struct AttnParams {
  const Group* groups;
  // paged context (null: contiguous): request r's context key j is pool row
  // block_table[r * max_pages + j / page_size] * page_size + j % page_size
  const int32_t* block_table;
  int max_pages, page_size;
  int64_t num_pages;
  const CtaRecord* cta_rec;  // balanced schedule
  uint32_t* hdr;
  float* part_o;
  float* part_ml;
  void* out;
  int hq, g, out_f32, causal, window, blk_tile;
  int grp_major;  // paged context K / V tiles laid out 8-row group by group in shared memory
  int balanced;  // stream-K schedule (else one whole group per CTA, round-robin)
  int grid;      // CTAs of the attention kernel (the combine kernel recomputes their ranges)
  float scale_log2;
};

struct TileInfo {
  int row;    // first source row (TMA outer coordinate)
  int valid;  // keys of this tile that belong to the request
  int j0;     // combined key index of the tile's first key
  bool blk;   // block-key tile (else context tile)
};

__device__ __forceinline__ TileInfo tile_info(const Group& U, int t, int blk_tile) {
  TileInfo ti;
  if (t < U.n_ctx_tiles) {
    const int k0 = U.ctx_lo + t * kTileKeys;
    ti.row = U.csl + k0;
    ti.valid = min(kTileKeys, U.clen - k0);
    ti.j0 = k0;
    ti.blk = false;
  } else {
    const int k0 = (t - U.n_ctx_tiles) * blk_tile;
    ti.row = U.qsl + k0;
    ti.valid = min(blk_tile, U.blen - k0);
    ti.j0 = U.clen + k0;
    ti.blk = true;
  }
  return ti;
}

// One segment of a CTA's work: key tiles [t0, t1) of one group.
struct Seg {
  Group grp;
  int t0, t1;
  int slot;       // partial slot (2 * cta + 0 for the CTA's first segment, + 1 otherwise)
  bool complete;  // the segment covers the whole group
};

// Walks the segments of this CTA. Every role of the CTA runs its own copy and sees the
// same sequence.
struct SegIter {
  const Group* groups;
  const Group* first;  // balanced: the first group, from the CTA record (shared memory)
  long long lo, hi;    // balanced: this CTA's tile range
  int ng, g, k;
  bool balanced;
  __device__ bool next(Seg& s) {
    if (balanced) {
      if (lo >= hi || g >= ng) return false;
      if (k == 0)
        s.grp = *first;
      else
        load_group(groups, g, s.grp);
      if (s.grp.start >= hi) return false;
      const long long st = s.grp.start;
      s.t0 = static_cast<int>((lo > st ? lo : st) - st);
      const long long end = st + s.grp.n;
      s.t1 = static_cast<int>((hi < end ? hi : end) - st);
      s.complete = s.t0 == 0 && s.t1 == s.grp.n;
      s.slot = 2 * static_cast<int>(blockIdx.x) + (k == 0 ? 0 : 1);
      ++k;
      ++g;
      return true;
    }
    if (g >= ng) return false;
    load_group(groups, g, s.grp);
    s.t0 = 0;
    s.t1 = s.grp.n;
    s.complete = true;
    s.slot = -1;
    g += gridDim.x;
    return true;
  }
  // Starts loading the descriptor the next call of next() reads (a segment switch then finds
  // it in L1 instead of waiting on L2 behind the K/V stream).
  __device__ void prefetch_next() const {
    if (g < ng) prefetch_l1(groups + g);
  }
};

// Producer of the paged instantiation (the whole warp 0). Q and block tiles come by TMA from
// lane 0. A context tile is one TMA box of page_size rows per page that holds its live keys,
// each at its rows of the tile: lane 0 posts the tile's byte count on the barrier and lane s
// issues the box of the tile's s-th page, so the boxes of a tile go out in parallel. Rows
// past the last such page are not loaded (the MMA and the softmax never read past the
// valid keys rounded up to 16, and the softmax zeroes the V rows in that gap). Page indices
// are loaded two tiles ahead.
template <int DH, int NK, int NV, int NQ, bool PRECISE>
__device__ __forceinline__ void produce_paged(const AttnParams& p, const CUtensorMap* tm_q, const CUtensorMap* tm_ql,
                                              const CUtensorMap* tm_kc, const CUtensorMap* tm_vc,
                                              const CUtensorMap* tm_kb, const CUtensorMap* tm_vb,
                                              const CUtensorMap* tm_kbl, SegIter it, uint32_t sbase, uint32_t bar0,
                                              volatile int* abort_flag, int lane) {
  const uint64_t pol_stream = l2_policy_evict_first();
  using L = Layout<DH, NK, NV, NQ, PRECISE>;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto wait0 = [&](uint32_t b, uint32_t parity) -> bool {  // lane 0 waits; every lane learns the outcome
    int r = 1;
    if (lane == 0) r = mbar_wait(b, parity, abort_flag) ? 1 : 0;
    return __shfl_sync(0xffffffffu, r, 0) != 0;
  };
  const int ps = p.page_size;
  uint32_t gk = 0, gv = 0;
  int iu = 0;
  bool ok = true;
  Seg sg;
  for (; ok && it.next(sg); ++iu) {
    if (lane == 0) it.prefetch_next();
    const Group& U = sg.grp;
    const int qb = iu % NQ;
    if (!(ok = wait0(bar(L::Q_EMPTY + qb), ((iu / NQ) & 1) ^ 1))) break;
    if (lane == 0) {
      const uint32_t q_rows = static_cast<uint32_t>(p.g * (kTileRows / p.g));
      mbar_arrive_expect_tx(bar(L::Q_FULL + qb), (PRECISE ? 2 : 1) * L::NB * q_rows * 128);
#pragma unroll
      for (int nb = 0; nb < L::NB; ++nb) {
        tma_load_4d(sbase + L::OFF_Q + qb * L::QBT + nb * (kTileRows * 128), tm_q, bar(L::Q_FULL + qb), nb * 64, 0,
                    U.kvh, U.qsl + U.tok0);
        if (PRECISE)
          tma_load_4d(sbase + L::OFF_Q + qb * L::QBT + L::QB + nb * (kTileRows * 128), tm_ql, bar(L::Q_FULL + qb),
                      nb * 64, 0, U.kvh, U.qsl + U.tok0);
      }
    }
    const int n = sg.t1 - sg.t0;
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(U.r) * p.max_pages;
    // lane s holds the index of the tile's s-th page
    auto tile_page = [&](int t) -> int {
      if (t >= sg.t1) return 0;
      const TileInfo ti = tile_info(U, t, p.blk_tile);
      if (ti.blk) return 0;
      const int nsub = (ti.valid + ps - 1) / ps;
      return lane < nsub ? __ldg(bt_row + ti.j0 / ps + lane) : 0;
    };
    auto issue = [&](int t, bool is_k, int pg) -> bool {
      const uint32_t cnt = is_k ? gk : gv;
      const int nst = is_k ? NK : NV;
      const int slot = static_cast<int>(cnt % nst);
      const uint32_t full = bar((is_k ? L::K_FULL : L::V_FULL) + slot);
      if (!wait0(bar((is_k ? L::K_EMPTY : L::V_EMPTY) + slot), ((cnt / nst) & 1) ^ 1)) return false;
      const TileInfo ti = tile_info(U, t, p.blk_tile);
      const uint32_t dst = sbase + (is_k ? L::OFF_K : L::OFF_V) + slot * L::KB;
      if (ti.blk) {
        if (lane == 0) {
          mbar_arrive_expect_tx(full, L::KB);
#pragma unroll
          for (int nb = 0; nb < L::NB; ++nb) {
            tma_load_3d(dst + nb * (kTileKeys * 128), is_k ? tm_kb : tm_vb, full, nb * 64, U.kvh, ti.row);
            if (PRECISE && is_k)  // a block tile holds 64 keys, hi in rows 0-63 and lo in rows 64-127
              tma_load_3d(dst + nb * (kTileKeys * 128) + 64 * 128, tm_kbl, full, nb * 64, U.kvh, ti.row);
          }
        }
      } else {
        const int nsub = (ti.valid + ps - 1) / ps;
        if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(nsub * ps * 128 * L::NB));
        if (lane < nsub && (pg < 0 || pg >= p.num_pages)) {  // reported; page 0 keeps the copy in bounds
          atomicOr(&p.hdr[0], kErrMetadata);
          pg = 0;
        }
        const void* map = is_k ? static_cast<const void*>(tm_kc) : static_cast<const void*>(tm_vc);
        if (p.grp_major) {
          // one box per lane: lane b copies page b whole, ps / 8 row groups
          if (lane < nsub)
            tma_load_5d_hint(dst + lane * (ps / 8) * kGroupBytes, map, full, 0, 0, 0, pg * (ps / 8), U.kvh,
                             pol_stream);
        } else {
          // one box per lane: lane b copies 64-column half b % NB of page b / NB
          const int my_page = __shfl_sync(0xffffffffu, pg, (lane / L::NB) & 31);
          if (lane < nsub * L::NB) {
            const int sp = lane / L::NB, nb = lane % L::NB;
            tma_load_3d_hint(dst + nb * (kTileKeys * 128) + sp * ps * 128, map, full, nb * 64, U.kvh, my_page * ps,
                             pol_stream);
          }
        }
      }
      if (is_k) ++gk; else ++gv;
      return true;
    };
    int pa = tile_page(sg.t0), pb = tile_page(sg.t0 + 1);
    if (!(ok = issue(sg.t0, true, pa))) break;
    for (int j = 0; j < n && ok; ++j) {
      const int pc = tile_page(sg.t0 + j + 2);
      if (j + 1 < n) ok = issue(sg.t0 + j + 1, true, pb);
      if (ok) ok = issue(sg.t0 + j, false, pa);
      pa = pb;
      pb = pc;
    }
  }
  if (!ok && lane == 0) atomicOr(&p.hdr[0], kErrTimeout);
  // every copy into shared memory has landed before the CTA can exit
  if (lane == 0) {
    for (int s = 0; s < NK; ++s)
      if (gk > static_cast<uint32_t>(s)) {
        const uint32_t last = ((gk - 1 - s) / NK) * NK + s;
        int dummy = 0;
        mbar_wait(bar(L::K_FULL + s), (last / NK) & 1, &dummy);
      }
    for (int s = 0; s < NV; ++s)
      if (gv > static_cast<uint32_t>(s)) {
        const uint32_t last = ((gv - 1 - s) / NV) * NV + s;
        int dummy = 0;
        mbar_wait(bar(L::V_FULL + s), (last / NV) & 1, &dummy);
      }
  }
}

#ifdef DFLASH_WAIT_TEST
// Test build only: (CTA, V tile count) of one V tile whose copy the producer withholds.
__device__ int2 g_withhold_v = {-1, -1};
#endif

template <int DH, int NK, int NV, int NQ, bool PRECISE, bool PAGED>
__global__ void __launch_bounds__(192, 1)
attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                 const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kb,
                 const __grid_constant__ CUtensorMap tm_vb, const __grid_constant__ CUtensorMap tm_ql,
                 const __grid_constant__ CUtensorMap tm_kbl, const __grid_constant__ AttnParams p) {
  using L = Layout<DH, NK, NV, NQ, PRECISE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(bar(L::K_FULL + i), 1);
      mbar_init(bar(L::K_EMPTY + i), 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(bar(L::V_FULL + i), 1);
      mbar_init(bar(L::V_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::Q_FULL + i), 1);
      // the MMA's last QK of the segment, and (staged epilogue) the four softmax warps once the
      // segment's output has left the buffer
      mbar_init(bar(L::Q_EMPTY + i), kStagedOut<NQ, PRECISE> ? 5 : 1);
      mbar_init(bar(L::S_FULL + i), 1);
      mbar_init(bar(L::S_EMPTY + i), 4);
      mbar_init(bar(L::P_FULL + i), 4);
      mbar_init(bar(L::P_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::O_FULL + i), 1);
      mbar_init(bar(L::O_EMPTY + i), 4);
    }
    mbar_init(bar(L::DRAIN), 1);
    *abort_flag = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
    tma_prefetch_desc(&tm_kb);
    tma_prefetch_desc(&tm_vb);
    if (PRECISE) {
      tma_prefetch_desc(&tm_ql);
      tma_prefetch_desc(&tm_kbl);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();  // group table and q^/k^ come from the prologue kernel
  grid_dependents_launch();
  // balanced: this CTA's record (first group, g0, lo, hi, ng); else g0 = blockIdx.x, ng
  int4* s_rec = reinterpret_cast<int4*>(smem + L::OFF_REC);
  if (p.balanced) {
    if (tid < 5) s_rec[tid] = reinterpret_cast<const int4*>(p.cta_rec + blockIdx.x)[tid];
  } else if (tid == 0) {
    s_rec[4] = make_int4(static_cast<int>(blockIdx.x), 0, 0, static_cast<int>(p.hdr[1]));
  }
  __syncthreads();
  auto make_iter = [&]() {
    SegIter it;
    it.groups = p.groups;
    it.first = reinterpret_cast<const Group*>(s_rec);
    it.lo = s_rec[4].y;
    it.hi = s_rec[4].z;
    it.g = s_rec[4].x;
    it.ng = s_rec[4].w;
    it.k = 0;
    it.balanced = p.balanced != 0;
    return it;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if constexpr (PAGED) {
      produce_paged<DH, NK, NV, NQ, PRECISE>(p, &tm_q, &tm_ql, &tm_kc, &tm_vc, &tm_kb, &tm_vb, &tm_kbl, make_iter(),
                                             sbase, bar0, abort_flag, lane);
    } else if (lane == 0) {
      uint32_t gk = 0, gv = 0;
      int iu = 0;
      bool ok = true;
      constexpr uint32_t q_box_bytes_per_row = 128;
      const uint64_t pol_stream = l2_policy_evict_first();
      SegIter it = make_iter();
      Seg sg;
      for (; ok && it.next(sg); ++iu) {
        it.prefetch_next();
        const Group& U = sg.grp;
        const int qb = iu % NQ;
        if (!(ok = mbar_wait(bar(L::Q_EMPTY + qb), ((iu / NQ) & 1) ^ 1, abort_flag))) break;
        // the Q box is G x (64 / G) rows whatever this unit's row count
        const uint32_t q_rows = static_cast<uint32_t>(p.g * (kTileRows / p.g));
        mbar_arrive_expect_tx(bar(L::Q_FULL + qb), (PRECISE ? 2 : 1) * L::NB * q_rows * q_box_bytes_per_row);
#pragma unroll
        for (int nb = 0; nb < L::NB; ++nb) {
          tma_load_4d(sbase + L::OFF_Q + qb * L::QBT + nb * (kTileRows * 128), &tm_q, bar(L::Q_FULL + qb), nb * 64, 0,
                      U.kvh, U.qsl + U.tok0);
          if (PRECISE)
            tma_load_4d(sbase + L::OFF_Q + qb * L::QBT + L::QB + nb * (kTileRows * 128), &tm_ql, bar(L::Q_FULL + qb),
                        nb * 64, 0, U.kvh, U.qsl + U.tok0);
        }
        const int n = sg.t1 - sg.t0;
        // context K/V tiles are read once: they should not push the split partials out of L2
        auto issue_k = [&](int t) -> bool {
          const int slot = static_cast<int>(gk % NK);
          if (!mbar_wait(bar(L::K_EMPTY + slot), ((gk / NK) & 1) ^ 1, abort_flag)) return false;
          const TileInfo ti = tile_info(U, t, p.blk_tile);
          mbar_arrive_expect_tx(bar(L::K_FULL + slot), L::KB);
          const void* map = ti.blk ? static_cast<const void*>(&tm_kb) : static_cast<const void*>(&tm_kc);
#pragma unroll
          for (int nb = 0; nb < L::NB; ++nb) {
            if (ti.blk)
              tma_load_3d(sbase + L::OFF_K + slot * L::KB + nb * (kTileKeys * 128), map, bar(L::K_FULL + slot),
                          nb * 64, U.kvh, ti.row);
            else
              tma_load_3d_hint(sbase + L::OFF_K + slot * L::KB + nb * (kTileKeys * 128), map, bar(L::K_FULL + slot),
                               nb * 64, U.kvh, ti.row, pol_stream);
            // precise mode: a block tile holds 64 keys, hi in rows 0-63 and lo in rows 64-127
            if (PRECISE && ti.blk)
              tma_load_3d(sbase + L::OFF_K + slot * L::KB + nb * (kTileKeys * 128) + 64 * 128, &tm_kbl,
                          bar(L::K_FULL + slot), nb * 64, U.kvh, ti.row);
          }
          ++gk;
          return true;
        };
        auto issue_v = [&](int t) -> bool {
          const int slot = static_cast<int>(gv % NV);
          if (!mbar_wait(bar(L::V_EMPTY + slot), ((gv / NV) & 1) ^ 1, abort_flag)) return false;
#ifdef DFLASH_WAIT_TEST
          if (static_cast<int>(blockIdx.x) == g_withhold_v.x && static_cast<int>(gv) == g_withhold_v.y) {
            ++gv;  // this tile's copy is never issued: its consumer's wait must run out
            return true;
          }
#endif
          const TileInfo ti = tile_info(U, t, p.blk_tile);
          mbar_arrive_expect_tx(bar(L::V_FULL + slot), L::KB);
          const void* map = ti.blk ? static_cast<const void*>(&tm_vb) : static_cast<const void*>(&tm_vc);
#pragma unroll
          for (int nb = 0; nb < L::NB; ++nb) {
            if (ti.blk)
              tma_load_3d(sbase + L::OFF_V + slot * L::KB + nb * (kTileKeys * 128), map, bar(L::V_FULL + slot),
                          nb * 64, U.kvh, ti.row);
            else
              tma_load_3d_hint(sbase + L::OFF_V + slot * L::KB + nb * (kTileKeys * 128), map, bar(L::V_FULL + slot),
                               nb * 64, U.kvh, ti.row, pol_stream);
          }
          ++gv;
          return true;
        };
        if (!(ok = issue_k(sg.t0))) break;
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) ok = issue_k(sg.t0 + j + 1);
          if (ok) ok = issue_v(sg.t0 + j);
        }
      }
      if (!ok) atomicOr(&p.hdr[0], kErrTimeout);
      // drain: wait (bounded) for every load this thread issued, so that no copy is
      // still writing shared memory when the CTA exits
      for (int s = 0; s < NK; ++s)
        if (gk > static_cast<uint32_t>(s)) {
          const uint32_t last = ((gk - 1 - s) / NK) * NK + s;  // last load into slot s
          int dummy = 0;
          mbar_wait(bar(L::K_FULL + s), (last / NK) & 1, &dummy);
        }
      for (int s = 0; s < NV; ++s)
        if (gv > static_cast<uint32_t>(s)) {
          const uint32_t last = ((gv - 1 - s) / NV) * NV + s;
          int dummy = 0;
          mbar_wait(bar(L::V_FULL + s), (last / NV) & 1, &dummy);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One pass over the CTA's tiles, segment after segment: S = Q K^T of the next tile is issued
    // before O += P V of the current one, across segment boundaries too (with two Q buffers),
    // so the next segment's first scores do not wait for the last V of this one. Segment iu
    // accumulates into O buffer iu & 1, so its first PV waits only for the epilogue of
    // segment iu - 2.
    if (lane == 0) {
      uint32_t gk = 0, gv = 0, gq = 0, gp = 0;  // K / V tiles consumed, QK / PV tiles issued
      bool ok = true;
      const uint32_t idesc_pv = umma_idesc_bf16(kTileRows, DH, 0, 1);
      SegIter it = make_iter();
      Seg cur, nxt;  // segment iu and, once fetched, segment iu + 1
      bool have_nxt = false;
      // S = Q K^T of tile j of segment iu (sg)
      auto issue_qk = [&](const Seg& sg, int iu, int j) -> bool {
        const Group& U = sg.grp;
        const int qb = iu % NQ;
        if (j == 0) {
          if (!mbar_wait(bar(L::Q_FULL + qb), (iu / NQ) & 1, abort_flag)) return false;
        }
        const uint32_t q_addr = sbase + L::OFF_Q + qb * L::QBT;
        const int sb = gq & 1;
        const int slot = static_cast<int>(gk % NK);
        if (!mbar_wait(bar(L::K_FULL + slot), (gk / NK) & 1, abort_flag)) return false;
        if (!mbar_wait(bar(L::S_EMPTY + sb), ((gq >> 1) & 1) ^ 1, abort_flag)) return false;
        tc_fence_after();
        const TileInfo ti = tile_info(U, sg.t0 + j, p.blk_tile);
        const int nq = min(kTileKeys, (ti.valid + 15) & ~15);
        const uint32_t idesc = umma_idesc_bf16(kTileRows, nq, 0, 0);
        const uint32_t k_addr = sbase + L::OFF_K + slot * L::KB;
        // group-major paged context tiles: column block nb at nb * 1 KB, 8-row groups 2 KB apart
        const bool gm = PAGED && p.grp_major && !ti.blk;
        const uint32_t k_nb = gm ? 1024 : kTileKeys * 128;
        const uint32_t k_sbo = gm ? kGroupBytes : 1024;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * (kTileRows * 128) + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * k_nb + (kk & 3) * 32;
          const uint64_t b = umma_desc_sw128(k_addr + ko, 16, k_sbo);
          umma_bf16_ss(tmem + sb * 128, umma_desc_sw128(q_addr + qo, 16, 1024), b, idesc, kk > 0 ? 1u : 0u);
          if (PRECISE) {
            // S = Q_hi K + Q_lo K (+ Q_hi K_lo on block tiles, whose keys are rounded here)
            umma_bf16_ss(tmem + sb * 128, umma_desc_sw128(q_addr + L::QB + qo, 16, 1024), b, idesc, 1u);
            if (ti.blk)
              umma_bf16_ss(tmem + sb * 128, umma_desc_sw128(q_addr + qo, 16, 1024),
                           umma_desc_sw128(k_addr + ko + 64 * 128, 16, 1024), idesc, 1u);
          }
        }
        umma_commit(bar(L::S_FULL + sb));
        umma_commit(bar(L::K_EMPTY + slot));
        if (j == sg.t1 - sg.t0 - 1) umma_commit(bar(L::Q_EMPTY + qb));
        ++gk;
        ++gq;
        return true;
      };
      bool have_cur = it.next(cur);
      if (have_cur) ok = issue_qk(cur, 0, 0);
      for (int iu = 0; ok && have_cur; ++iu) {
        const Seg& sg = cur;
        const int n = sg.t1 - sg.t0;
        const uint32_t o_col = 256 + static_cast<uint32_t>((iu & 1) * DH);
        bool next_issued = false;
        it.prefetch_next();
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) {
            if (!(ok = issue_qk(sg, iu, j + 1))) break;
          } else if (NQ > 1 && (have_nxt = it.next(nxt))) {
            // the next segment's first QK before this segment's last PV
            if (!(ok = issue_qk(nxt, iu + 1, 0))) break;
            next_issued = true;
          }
          const int pb = gp & 1;
          const int vslot = static_cast<int>(gv % NV);
          if (!(ok = mbar_wait(bar(L::P_FULL + pb), (gp >> 1) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(bar(L::V_FULL + vslot), (gv / NV) & 1, abort_flag))) break;
          if (j == 0 && !(ok = mbar_wait(bar(L::O_EMPTY + (iu & 1)), ((iu >> 1) & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          const TileInfo ti = tile_info(sg.grp, sg.t0 + j, p.blk_tile);
          const int ksteps = (ti.valid + 15) >> 4;
          const uint32_t p_addr = sbase + L::OFF_P + pb * L::PBT;
          const uint32_t v_addr = sbase + L::OFF_V + vslot * L::KB;
          // group-major paged context tiles: 16 keys = two groups, column blocks 1 KB apart
          const bool gm = PAGED && p.grp_major && !ti.blk;
          const uint32_t v_step = gm ? 2 * kGroupBytes : 16 * 128;
          const uint32_t v_lbo = gm ? 1024 : kTileKeys * 128;
          const uint32_t v_sbo = gm ? kGroupBytes : 1024;
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint32_t po = (kk >> 2) * (kTileRows * 128) + (kk & 3) * 32;
            const uint64_t b = umma_desc_sw128(v_addr + kk * v_step, v_lbo, v_sbo);
            umma_bf16_ss(tmem + o_col, umma_desc_sw128(p_addr + po, 16, 1024), b, idesc_pv,
                         (j > 0 || kk > 0) ? 1u : 0u);
            if (PRECISE) umma_bf16_ss(tmem + o_col, umma_desc_sw128(p_addr + L::PB + po, 16, 1024), b, idesc_pv, 1u);
          }
          umma_commit(bar(L::V_EMPTY + vslot));
          umma_commit(bar(L::P_EMPTY + pb));
          ++gv;
          ++gp;
        }
        if (!ok) break;
        umma_commit(bar(L::O_FULL + (iu & 1)));
        // one Q buffer: the next segment's Q is loaded after this segment's last QK, so its
        // first QK comes after the last PV
        if (NQ == 1) have_nxt = it.next(nxt);
        if (!next_issued && have_nxt) ok = issue_qk(nxt, iu + 1, 0);
        have_cur = have_nxt;
        if (have_cur) cur = nxt;
      }
      if (!ok) atomicOr(&p.hdr[0], kErrTimeout);
      // let every issued MMA finish before the CTA releases tensor memory
      umma_commit(bar(L::DRAIN));
      int dummy = 0;
      mbar_wait(bar(L::DRAIN), 0, &dummy);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int sp = warp & 3;                      // TMEM sub-partition of this warp
    const int rho = 16 * sp + (lane & 15);        // query row of this thread
    const int half = lane >> 4;                   // key columns [64*half, 64*half + 64)
    const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
    const float sl2 = p.scale_log2;
    uint32_t gj = 0, gv = 0;
    int iu = 0;
    bool ok = true;
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      int r = 1;
      if (lane == 0) r = mbar_wait(b, parity, abort_flag) ? 1 : 0;
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    // A segment's epilogue runs once the next segment's first P is written (the MMA meanwhile
    // starts the next segment in the other O buffer), or after the last segment.
    struct Pending {
      int row;      // output row (token * Hq + head) of this thread (complete segment)
      float m, l;
      int state;    // bit 0 valid, bit 1 row ok, bit 2 complete, bits 3..: segment index
      __device__ bool valid() const { return state & 1; }
    } pend;
    pend.state = 0;
    constexpr int CH = DH / 2 / 32;  // 32-column chunks per half row of O
    auto epilogue = [&](const Pending& e) -> bool {
      const int e_iu = e.state >> 3;
      if (!wait_warp(bar(L::O_FULL + (e_iu & 1)), (e_iu >> 1) & 1)) return false;
      tc_fence_after();
      uint32_t o[CH][32];
      const uint32_t o_col = 256 + static_cast<uint32_t>((e_iu & 1) * DH);
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) tmem_ld_16x32bx2_x32<DH / 2>(tmem + lane_base + o_col + ch * 32, o[ch]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::O_EMPTY + (e_iu & 1)));
      const float l_tot = e.l + __shfl_xor_sync(0xffffffffu, e.l, 16);
      const bool row_ok = (e.state & 2) != 0;
      if ((e.state & 4) && kStagedOut<NQ, PRECISE>) {
        // bf16 rows through the segment's Q buffer, 128-byte swizzled: this warp's 16 rows at
        // sp * 16 rows; 16-byte chunk k of row r at chunk position k ^ (r & 7)
        const float inv = l_tot > 0.0f ? 1.0f / l_tot : 0.0f;
        constexpr int CPRW = DH * 2 / 16;  // 16-byte chunks per row
        uint8_t* stg = smem + L::OFF_Q + (e_iu % NQ) * L::QBT + sp * (16 * DH * 2);
        const int r16 = lane & 15;
#pragma unroll
        for (int ch = 0; ch < CH; ++ch)
#pragma unroll
          for (int x = 0; x < 32; x += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[ch][x]) * inv, __uint_as_float(o[ch][x + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[ch][x + 2]) * inv, __uint_as_float(o[ch][x + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[ch][x + 4]) * inv, __uint_as_float(o[ch][x + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[ch][x + 6]) * inv, __uint_as_float(o[ch][x + 7]) * inv);
            const int k = half * (CPRW / 2) + ch * 4 + x / 8;
            *reinterpret_cast<uint4*>(stg + r16 * (DH * 2) + ((k ^ (r16 & 7)) << 4)) = v;
          }
        __syncwarp();
        // read back a row per half-warp (two rows per step at Dh = 128, four at Dh = 64)
        constexpr int RPI = 32 / CPRW;
#pragma unroll
        for (int i = 0; i < 16 / RPI; ++i) {
          const int r = i * RPI + lane / CPRW, c = lane % CPRW;
          const int row_g = __shfl_sync(0xffffffffu, e.row, r);
          const int ok_r = __shfl_sync(0xffffffffu, row_ok ? 1 : 0, r);
          const uint4 v = *reinterpret_cast<const uint4*>(stg + r * (DH * 2) + ((c ^ (r & 7)) << 4));
          if (ok_r) *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(row_g) * DH + c * 8) = v;
        }
        __syncwarp();
      } else if (!row_ok) {
        // no output row (a query tile's rows past its group's last token)
      } else if (e.state & 4) {
        const float inv = l_tot > 0.0f ? 1.0f / l_tot : 0.0f;
        if (p.out_f32) {
          float* dst = reinterpret_cast<float*>(p.out) + static_cast<int64_t>(e.row) * DH + half * (DH / 2);
#pragma unroll
          for (int ch = 0; ch < CH; ++ch)
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              *reinterpret_cast<float4*>(dst + ch * 32 + x) =
                  make_float4(__uint_as_float(o[ch][x]) * inv, __uint_as_float(o[ch][x + 1]) * inv,
                              __uint_as_float(o[ch][x + 2]) * inv, __uint_as_float(o[ch][x + 3]) * inv);
        } else {
          uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(e.row) * DH + half * (DH / 2);
#pragma unroll
          for (int ch = 0; ch < CH; ++ch)
#pragma unroll
            for (int x = 0; x < 32; x += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[ch][x]) * inv, __uint_as_float(o[ch][x + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(o[ch][x + 2]) * inv, __uint_as_float(o[ch][x + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(o[ch][x + 4]) * inv, __uint_as_float(o[ch][x + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(o[ch][x + 6]) * inv, __uint_as_float(o[ch][x + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + ch * 32 + x) = v;
            }
        }
      } else {
        // kept in L2 for the combine pass, which reads them after the streaming
        const uint64_t pol_keep = l2_policy_evict_last();
        const int pslot = 2 * static_cast<int>(blockIdx.x) + (e_iu == 0 ? 0 : 1);  // first segment, or later
        // the slot is laid out in the order the threads hold it (part_o_index): every store
        // instruction of the warp writes 512 contiguous bytes
        float* dst = p.part_o + (static_cast<int64_t>(pslot) * kTileRows * DH) + part_o_index<DH>(sp, 0, lane) * 4;
#pragma unroll
        for (int ch = 0; ch < CH; ++ch)
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            st_global_v4_hint(dst + (ch * 8 + x / 4) * 32 * 4,
                              make_float4(__uint_as_float(o[ch][x]), __uint_as_float(o[ch][x + 1]),
                                          __uint_as_float(o[ch][x + 2]), __uint_as_float(o[ch][x + 3])),
                              pol_keep);
        if (half == 0)
          st_global_v2_hint(p.part_ml + (static_cast<int64_t>(pslot) * kTileRows + rho) * 2, e.m, l_tot, pol_keep);
      }
      if (kStagedOut<NQ, PRECISE> && lane == 0) mbar_arrive(bar(L::Q_EMPTY + (e_iu % NQ)));
      return true;
    };
    // One pass per segment, plus a last one without tiles for the last segment's epilogue, so
    // that the tile body and the epilogue each appear once in the code (cold code is fetched
    // from memory the first time it runs).
    SegIter it = make_iter();
    Seg sg;
    bool have = it.next(sg);
    for (; ok && (have || pend.valid()); ++iu) {
      if (have && lane == 0) it.prefetch_next();
      const Group& U = sg.grp;
      const int n = have ? sg.t1 - sg.t0 : 0;
      const bool row_ok = rho < U.rows;
      const int b = U.tok0 + rho / p.g;        // block index of this row
      const int i = U.clen + b;                // combined query index
      int jlo = 0, jhi = U.clen + U.blen - 1;
      if (p.causal) {
        jhi = i;
        if (p.window > 0) jlo = max(0, i - p.window + 1);
      }
      if (!row_ok) {
        jlo = 1;
        jhi = 0;
      }
      float m_used = -INFINITY, l = 0.0f;
      for (int j = 0; j < (n > 0 ? n : 1); ++j) {
       if (j < n) {
        const uint32_t g = gj + j;
        const int sb = g & 1;
        const TileInfo ti = tile_info(U, sg.t0 + j, p.blk_tile);
        if (!(ok = wait_warp(bar(L::S_FULL + sb), (g >> 1) & 1))) break;
        tc_fence_after();
        uint32_t sr[64];
        {
          uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
          uint32_t (&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
          tmem_ld_16x32bx2_x32<64>(tmem + lane_base + sb * 128, a);
          tmem_ld_16x32bx2_x32<64>(tmem + lane_base + sb * 128 + 32, c);
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::S_EMPTY + sb));
        // scale to base 2 and mask
        const int col0 = 64 * half;
        const int jbase = ti.j0 + col0;
        const bool full_tile = ti.valid == kTileKeys && ti.j0 >= jlo && ti.j0 + kTileKeys - 1 <= jhi;
        // the running maximum is taken over the raw scores (the scale is positive); masked keys
        // become -inf in place
        float* x = reinterpret_cast<float*>(sr);
        if (!full_tile) {
          const int c_lo = max(jlo - jbase, 0);
          const int c_hi = min(jhi - jbase, ti.valid - col0 - 1);
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = (c >= c_lo && c <= c_hi) ? x[c] : -INFINITY;
        }
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c += 2) mt = fmax3(mt, x[c], x[c + 1]);
        mt *= sl2;
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        float alpha = 1.0f;
        bool rescale = false;
        if (j == 0) {
          m_used = mt;
        } else if (mt > m_used + 8.0f) {
          if (m_used != -INFINITY) {
            alpha = ex2_approx(m_used - mt);
            rescale = true;
          }
          m_used = mt;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O must hold PV of tile j-1 before it is rescaled
          if (!(ok = wait_warp(bar(L::P_EMPTY + ((g - 1) & 1)), ((g - 1) >> 1) & 1))) break;
          tc_fence_after();
          l *= alpha;
#pragma unroll
          for (int ch = 0; ch < CH; ++ch) {
            uint32_t o[32];
            const uint32_t o_addr = tmem + lane_base + 256 + static_cast<uint32_t>((iu & 1) * DH) + ch * 32;
            tmem_ld_16x32bx2_x32<DH / 2>(o_addr, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_16x32bx2_x32<DH / 2>(o_addr, o);
          }
          tmem_wait_st();
        }
        const float m_eff = m_used == -INFINITY ? 0.0f : m_used;
        // exponent s * scale - m for two keys per instruction; the weight sums two lanes wide
        const uint64_t sl2x2 = f32x2(sl2, sl2), negm = f32x2(-m_eff, -m_eff);
        uint32_t pk[32];
        uint32_t pl[PRECISE ? 32 : 1];
        uint64_t lsum2 = f32x2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float a0, a1;
          f32x2_split(fma_f32x2(f32x2(x[c], x[c + 1]), sl2x2, negm), a0, a1);
          const float p0 = ex2_approx(a0);
          const float p1 = ex2_approx(a1);
          const uint32_t v = pack_bf16x2(p0, p1);
          pk[c / 2] = v;
          if (PRECISE) {
            // P = P_hi + P_lo; l sums the unrounded weights
            pl[c / 2] = pack_bf16x2(p0 - bf16lo_to_f32(v), p1 - bf16hi_to_f32(v));
            lsum2 = add_f32x2(lsum2, f32x2(p0, p1));
          } else {
            lsum2 = add_f32x2(lsum2, f32x2(bf16lo_to_f32(v), bf16hi_to_f32(v)));  // exactly the weights PV uses
          }
        }
        {
          float s0, s1;
          f32x2_split(lsum2, s0, s1);
          l += s0 + s1;
        }
        // the P buffer is free once PV of tile g-2 has completed
        if (!(ok = wait_warp(bar(L::P_EMPTY + sb), ((g >> 1) & 1) ^ 1))) break;
        {
          uint8_t* prow = smem + L::OFF_P + sb * L::PBT + half * (kTileRows * 128) + rho * 128;
#pragma unroll
          for (int chn = 0; chn < 8; ++chn) {
            uint4 v = make_uint4(pk[4 * chn], pk[4 * chn + 1], pk[4 * chn + 2], pk[4 * chn + 3]);
            *reinterpret_cast<uint4*>(prow + ((chn ^ (rho & 7)) << 4)) = v;
            if (PRECISE) {
              uint4 w = make_uint4(pl[4 * chn], pl[4 * chn + 1], pl[4 * chn + 2], pl[4 * chn + 3]);
              *reinterpret_cast<uint4*>(prow + L::PB + ((chn ^ (rho & 7)) << 4)) = w;
            }
          }
        }
        if (ti.valid & 15) {
          // keys [valid, valid rounded up to 16) enter the last PV step with P = 0;
          // zero those V rows so that whatever the copy brought in cannot make a NaN
          const uint32_t vg = gv + j;
          const int vslot = static_cast<int>(vg % NV);
          if (!(ok = wait_warp(bar(L::V_FULL + vslot), (vg / NV) & 1))) break;
          const int r0 = ti.valid, r1 = (ti.valid + 15) & ~15;
          const int wg_tid = tid - 64;
          const int chunks = (r1 - r0) * L::NB * 8;  // 16-byte chunks to clear
          for (int c = wg_tid; c < chunks; c += 128) {
            const int row = r0 + c / (L::NB * 8);
            const int rem = c % (L::NB * 8);
            const int nb = rem / 8, chn = rem % 8;
            const int off = (PAGED && p.grp_major && !ti.blk)
                                ? (row / 8) * static_cast<int>(kGroupBytes) + nb * 1024 + (row % 8) * 128
                                : nb * (kTileKeys * 128) + row * 128;
            *reinterpret_cast<uint4*>(smem + L::OFF_V + vslot * L::KB + off + chn * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::P_FULL + sb));
       }
        if (j == 0 && pend.valid()) {  // the previous segment's epilogue, now that this one has started
          if (!(ok = epilogue(pend))) break;
          pend.state = 0;
        }
      }
      if (!ok) break;
      if (!have) continue;
      // ---------------------------------------------------------- epilogue (deferred)
      pend.state = 1 | (row_ok ? 2 : 0) | (sg.complete ? 4 : 0) | (iu << 3);
      pend.m = m_used;
      pend.l = l;
      pend.row = (U.qsl + b) * p.hq + U.kvh * p.g + rho % p.g;
      gj += n;
      gv += n;
      have = it.next(sg);
    }
    if (!ok) atomicOr(&p.hdr[0], kErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================ kernel C
// One block per CTA boundary b (between CTAs b and b+1 of the attention kernel) and
// 16-row slice: the group holding the boundary's tile is CTA b+1's first group, split
// if it starts before CTA b+1's first tile. A group split by several boundaries is merged
// by the block of its first one. The records come from the prologue, which completed
// before the attention kernel passed its own dependency wait and let this grid launch,
// so they are read before this grid's wait, which only the partials need.
template <int DH>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnParams p) {
  const int b = blockIdx.x;  // boundary between CTAs b and b + 1
  Group G;
  int lo1;
  {
    const CtaRecord* rec = p.cta_rec + b + 1;
    const int4* src = reinterpret_cast<const int4*>(&rec->first);
    int4* dst = reinterpret_cast<int4*>(&G);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = __ldcg(src + i);
    lo1 = __ldcg(&rec->lo);
  }
  const long long tt = static_cast<long long>(__ldcg(p.hdr + 2));
  const long long grid = p.grid;
  const long long lo0 = __ldcg(&p.cta_rec[b].lo);  // CTA b's first tile
  // split at this boundary, and not at an earlier one
  const bool mine = tt > 0 && G.start < lo1 && G.start >= lo0;
  // contributors: CTAs ca = b .. cb, the last one being the last CTA whose first tile lies in
  // the group (no CTA between is empty: empty CTAs only follow the last tile)
  const long long ca = b;
  long long cb = b + 1;
  if (mine) {
    const long long gend = static_cast<long long>(G.start) + G.n;
    while (cb + 1 < grid && __ldcg(&p.cta_rec[cb + 1].lo) < gend) ++cb;
  }
  grid_dependency_wait();
  if (!mine) return;
  // the group is CTA b's first segment iff it starts at lo0
  const bool ca_first = G.start == lo0;
  // Block y covers rows [16y, 16y + 16): thread t merges the 4-float groups k0 = t / 32 and
  // k0 + DH / 16 that lane t % 32 of TMEM sub-partition y stored (part_o_index), so that every
  // load of a warp reads 512 contiguous bytes.
  constexpr int kMaxBatch = 2;  // contributors whose loads are in flight together
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int rho = 16 * static_cast<int>(blockIdx.y) + (lane & 15);
  if (rho >= G.rows) return;
  const int k0 = static_cast<int>(threadIdx.x >> 5);
  // running merge: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, contributors in batches
  float M = -INFINITY, L = 0.0f;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (long long c = ca; c <= cb; c += kMaxBatch) {
    float2 ml[kMaxBatch];
    float4 oa[kMaxBatch], ob[kMaxBatch];
#pragma unroll
    for (int i = 0; i < kMaxBatch; ++i) {
      const long long cc = c + i;
      if (cc <= cb) {
        const long long slot = 2 * cc + ((cc == ca && !ca_first) ? 1 : 0);
        ml[i] = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (slot * kTileRows + rho) * 2));
        const float4* src =
            reinterpret_cast<const float4*>(p.part_o + slot * kTileRows * DH) + part_o_index<DH>(blockIdx.y, k0, lane);
        oa[i] = __ldcg(src);
        ob[i] = __ldcg(src + (DH / 16) * 32);
      } else {
        ml[i] = make_float2(-INFINITY, 0.0f);
        oa[i] = ob[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
    float Mn = M;
#pragma unroll
    for (int i = 0; i < kMaxBatch; ++i) Mn = fmaxf(Mn, ml[i].x);
    if (Mn == -INFINITY) continue;
    const float r = M == -INFINITY ? 0.0f : ex2_approx(M - Mn);
    L *= r;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= r;
#pragma unroll
    for (int i = 0; i < kMaxBatch; ++i) {
      const float w = ml[i].x == -INFINITY ? 0.0f : ex2_approx(ml[i].x - Mn);
      L += w * ml[i].y;
      acc[0] += w * oa[i].x; acc[1] += w * oa[i].y; acc[2] += w * oa[i].z; acc[3] += w * oa[i].w;
      acc[4] += w * ob[i].x; acc[5] += w * ob[i].y; acc[6] += w * ob[i].z; acc[7] += w * ob[i].w;
    }
    M = Mn;
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  const int64_t tok = G.qsl + G.tok0 + rho / p.g;
  const int head = G.kvh * p.g + rho % p.g;
  const int64_t col_a = (lane >> 4) * (DH / 2) + 4 * k0;  // columns of the first group
  const int64_t col_b = col_a + 4 * (DH / 16);             // and of the second
  if (p.out_f32) {
    float* row = reinterpret_cast<float*>(p.out) + (tok * p.hq + head) * DH;
    *reinterpret_cast<float4*>(row + col_a) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<float4*>(row + col_b) = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  } else {
    uint16_t* row = reinterpret_cast<uint16_t*>(p.out) + (tok * p.hq + head) * DH;
    *reinterpret_cast<uint2*>(row + col_a) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                        pack_bf16x2(acc[2] * inv, acc[3] * inv));
    *reinterpret_cast<uint2*>(row + col_b) = make_uint2(pack_bf16x2(acc[4] * inv, acc[5] * inv),
                                                        pack_bf16x2(acc[6] * inv, acc[7] * inv));
  }
}

// ================================================================ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// rank-3 view {dh, heads, rows} of a [rows, heads, dh] bf16 tensor, box {64, 1, box_rows}
static bool encode_rows_map(CUtensorMap* m, const void* base, int dh, int heads, int64_t rows, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dh), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dh) * 2, static_cast<cuuint64_t>(dh) * heads * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Group-major view of a paged pool [rows, heads, dh] with dh = 128: dimensions {64 columns,
// 8 rows, 2 column blocks, rows / 8 groups, heads} (strides: row 2 KB-ish, column block 128 B,
// group 8 rows, head dh * 2), box {64, 8, 2, page_size / 8, 1}: one box lands as the page's
// 8-row groups, each as its two column blocks one after the other.
static bool encode_group_major_map(CUtensorMap* m, const void* base, int dh, int heads, int64_t rows, int page_size) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(dh) * heads * 2;
  cuuint64_t dims[5] = {64, 8, static_cast<cuuint64_t>(dh / 64), static_cast<cuuint64_t>(rows > 0 ? rows / 8 : 1),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[4] = {row_bytes, 128, 8 * row_bytes, static_cast<cuuint64_t>(dh) * 2};
  cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(dh / 64), static_cast<cuuint32_t>(page_size / 8), 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// rank-4 view {dh, g, hkv, tokens} of q^ [tokens, hkv*g, dh], box {64, g, 1, tpq}
static bool encode_q_map(CUtensorMap* m, const void* base, int dh, int g, int hkv, int64_t tokens, int tpq) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(dh), static_cast<cuuint64_t>(g), static_cast<cuuint64_t>(hkv),
                        static_cast<cuuint64_t>(tokens > 0 ? tokens : 1)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(dh) * 2, static_cast<cuuint64_t>(dh) * g * 2,
                           static_cast<cuuint64_t>(dh) * g * hkv * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(tpq)};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

WorkspacePlan plan_workspace(int num_reqs, int64_t total_q, int hq, int hkv, int dh, int64_t total_ctx,
                             int max_ctx_len, int max_block_len, int window, int causal, int precise, int flags,
                             int num_sms) {
  WorkspacePlan w{};
  const int g = hq / hkv;
  w.tpq = kTileRows / g;
  w.qt_max = max_block_len > 0 ? (max_block_len + w.tpq - 1) / w.tpq : 0;
  int ctx_tiles_max = (max_ctx_len + kTileKeys - 1) / kTileKeys;
  if (causal && window > 0) ctx_tiles_max = std::min(ctx_tiles_max, (window - 1 + kTileKeys - 1) / kTileKeys + 1);
  const int blk_tile = precise ? 64 : kTileKeys;
  const int blk_tiles_max = (max_block_len + blk_tile - 1) / blk_tile;
  const int n_max = std::max(1, ctx_tiles_max + blk_tiles_max);
  // key tiles of all groups: an upper bound from the segment capacities and the lengths
  double per_head = static_cast<double>(total_ctx) / kTileKeys + static_cast<double>(num_reqs) * (1 + blk_tiles_max);
  per_head = std::min(per_head, static_cast<double>(num_reqs) * n_max);
  w.tiles_bound = static_cast<double>(hkv) * std::max(1, w.qt_max) * per_head;
  w.groups_max = std::max(1, num_reqs * hkv * std::max(1, w.qt_max));
  w.balanced = (flags & 2) == 0;  // DFLASH_FLAG_NO_SPLIT selects whole groups per CTA
  if (w.balanced) {
    // every CTA should stream at least kMinTilesPerCta tiles so that its set-up is amortised
    // (4 measured faster than 8 on the Qwen3-0.6B-shaped layer: more SMs stream, and the
    // per-SM bandwidth, not the chip's, is what a CTA gets)
    constexpr double kMinTilesPerCta = 4.0;
    w.grid = static_cast<int>(std::min<double>(num_sms, std::max(1.0, std::ceil(w.tiles_bound / kMinTilesPerCta))));
  } else {
    w.grid = std::min(num_sms, w.groups_max);
  }
  w.grid = std::max(1, w.grid);
  w.parts = w.balanced ? 2 * w.grid : 0;
  size_t off = 0;
  w.hdr = off;
  off += 256;
  w.q_hat = off;
  off += align256(static_cast<size_t>(total_q) * hq * dh * 2);
  w.q_lo = off;
  if (precise) off += align256(static_cast<size_t>(total_q) * hq * dh * 2);
  w.k_hat = off;
  off += align256(static_cast<size_t>(total_q) * hkv * dh * 2);
  w.k_lo = off;
  if (precise) off += align256(static_cast<size_t>(total_q) * hkv * dh * 2);
  w.groups = off;
  off += align256(static_cast<size_t>(w.groups_max) * sizeof(Group));
  w.cta_rec = off;
  if (w.balanced) off += align256(static_cast<size_t>(w.grid) * sizeof(CtaRecord));
  w.part_o = off;
  off += align256(static_cast<size_t>(w.parts) * kTileRows * dh * 4);
  w.part_ml = off;
  off += align256(static_cast<size_t>(w.parts) * kTileRows * 2 * 4);
  w.total = off;
  return w;
}

template <int DH, int NK, int NV, int NQ, bool PRECISE, bool PAGED>
static cudaError_t launch_b(const CUtensorMap& tq, const CUtensorMap& tkc, const CUtensorMap& tvc,
                            const CUtensorMap& tkb, const CUtensorMap& tvb, const CUtensorMap& tql,
                            const CUtensorMap& tkbl, const AttnParams& ap, int grid, cudaStream_t stream) {
  using L = Layout<DH, NK, NV, NQ, PRECISE>;
  static_assert(L::ALLOC <= 232448, "shared memory plan exceeds the per-block limit");
  auto kern = attention_kernel<DH, NK, NV, NQ, PRECISE, PAGED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tkc, tvc, tkb, tvb, tql, tkbl, ap);
}

template <int DH>
static cudaError_t launch_c(const AttnParams& ap, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, kTileRows / 16);
  cfg.blockDim = dim3(16 * DH / 8);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<DH>, ap);
}

cudaError_t launch_attention(const AttnHost& h, cudaStream_t stream, char* msg, size_t msg_len) {
  if (h.total_q <= 0 || h.num_reqs <= 0) return cudaSuccess;
  // ---- A: prologue
  PrologueParams pp{};
  pp.job.nparts = 2;
  pp.job.part[0] = NormRopePart{h.q, h.q_norm_w, h.q_hat, h.precise ? h.q_lo : nullptr, nullptr, nullptr, h.hq};
  pp.job.part[1] = NormRopePart{h.k_blk, h.k_norm_w, h.k_hat, h.precise ? h.k_lo : nullptr, nullptr, nullptr, h.hkv};
  pp.job.n_tok = h.total_q;
  pp.job.pos = h.positions;
  pp.job.slot = nullptr;
  pp.job.capacity = h.total_q;
  pp.job.eps = h.eps;
  pp.job.err = h.ws_hdr;
  pp.job.turns = h.turns;
  pp.qsl = h.qsl;
  pp.csl = h.csl;
  pp.clen = h.clen;
  pp.groups = h.groups;
  pp.cta_rec = h.balanced ? h.cta_rec : nullptr;
  pp.grid_b = h.grid;
  pp.hdr = h.ws_hdr;
  pp.total_q = h.total_q;
  pp.total_ctx = h.total_ctx;
  pp.num_reqs = h.num_reqs;
  pp.hkv = h.hkv;
  pp.g = h.g;
  pp.tpq = h.tpq;
  pp.causal = h.causal;
  pp.window = h.window;
  pp.groups_max = h.groups_max;
  pp.max_ctx_len = h.max_ctx_len;
  pp.max_block_len = h.max_block_len;
  pp.blk_tile = h.precise ? 64 : kTileKeys;
  pp.paged = h.paged ? 1 : 0;
  pp.page_size = h.paged ? h.page_size : 1;
  pp.paged_cap = h.paged ? h.max_pages * h.page_size : 0;
  cudaError_t e = cudaSuccess;
  int64_t nr_blocks = (h.total_q * norm_rope_items_per_token(pp.job, h.dh) + 7) / 8;
  nr_blocks = std::min<int64_t>(nr_blocks, static_cast<int64_t>(h.num_sms) * 3 - kTableBlocks);  // all co-resident
  const unsigned grid_a = static_cast<unsigned>(kTableBlocks + nr_blocks);
  if (h.dh == 128)
    prologue_kernel<128><<<grid_a, 256, 0, stream>>>(pp);
  else
    prologue_kernel<64><<<grid_a, 256, 0, stream>>>(pp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // ---- tensor maps
  CUtensorMap tq, tkc, tvc, tkb, tvb, tql, tkbl;
  const void* ctx_k = h.total_ctx > 0 ? static_cast<const void*>(h.ctx_k) : static_cast<const void*>(h.q_hat);
  const void* ctx_v = h.total_ctx > 0 ? static_cast<const void*>(h.ctx_v) : static_cast<const void*>(h.q_hat);
  const int64_t ctx_rows = h.total_ctx > 0 ? h.total_ctx : 1;
  const bool grp_major = h.paged && h.dh == 128;
  bool ok = encode_q_map(&tq, h.q_hat, h.dh, h.g, h.hkv, h.total_q, h.tpq) &&
            (grp_major ? encode_group_major_map(&tkc, ctx_k, h.dh, h.hkv, ctx_rows, h.page_size) &&
                             encode_group_major_map(&tvc, ctx_v, h.dh, h.hkv, ctx_rows, h.page_size)
                       : encode_rows_map(&tkc, ctx_k, h.dh, h.hkv, ctx_rows, h.paged ? h.page_size : kTileKeys) &&
                             encode_rows_map(&tvc, ctx_v, h.dh, h.hkv, ctx_rows, h.paged ? h.page_size : kTileKeys)) &&
            encode_rows_map(&tkb, h.k_hat, h.dh, h.hkv, h.total_q, h.precise ? 64 : kTileKeys) &&
            encode_rows_map(&tvb, h.v_blk, h.dh, h.hkv, h.total_q, kTileKeys);
  if (ok && h.precise)
    ok = encode_q_map(&tql, h.q_lo, h.dh, h.g, h.hkv, h.total_q, h.tpq) &&
         encode_rows_map(&tkbl, h.k_lo, h.dh, h.hkv, h.total_q, 64);
  if (!h.precise) {
    tql = tq;
    tkbl = tkb;
  }
  if (!ok) {
    std::snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (driver entry point or tensor layout)");
    return cudaErrorInvalidValue;
  }
  AttnParams ap{};
  ap.groups = h.groups;
  ap.cta_rec = h.cta_rec;
  ap.hdr = h.ws_hdr;
  ap.part_o = h.part_o;
  ap.part_ml = h.part_ml;
  ap.out = h.out;
  ap.hq = h.hq;
  ap.g = h.g;
  ap.out_f32 = h.out_f32;
  ap.causal = h.causal;
  ap.window = h.window;
  ap.scale_log2 = h.scale_log2;
  ap.blk_tile = h.precise ? 64 : kTileKeys;
  ap.block_table = h.paged ? h.block_table : nullptr;
  ap.max_pages = h.max_pages;
  ap.page_size = h.paged ? h.page_size : kTileKeys;
  ap.grp_major = grp_major ? 1 : 0;
  ap.num_pages = h.paged ? h.total_ctx / h.page_size : 0;
  ap.balanced = h.balanced ? 1 : 0;
  ap.grid = h.grid;
  const int grid_b = h.grid;
  // ---- B: attention
  // K/V rings: Dh = 128, 3 K + 2 V stages of 32 KB (2 + 2 with the hi/lo halves of precise
  // mode); Dh = 64, 4 + 4 (3 + 3). Paged contexts have their own instantiations, so that the
  // contiguous kernels carry no paged code.
  if (h.paged) {
    if (h.dh == 128)
      e = h.precise ? launch_b<128, 2, 2, 1, true, true>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream)
                    : launch_b<128, 3, 2, 2, false, true>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream);
    else
      e = h.precise ? launch_b<64, 3, 3, 2, true, true>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream)
                    : launch_b<64, 4, 4, 2, false, true>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream);
  } else {
    if (h.dh == 128)
      e = h.precise ? launch_b<128, 2, 2, 1, true, false>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream)
                    : launch_b<128, 3, 2, 2, false, false>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream);
    else
      e = h.precise ? launch_b<64, 3, 3, 2, true, false>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream)
                    : launch_b<64, 4, 4, 2, false, false>(tq, tkc, tvc, tkb, tvb, tql, tkbl, ap, grid_b, stream);
  }
  if (e != cudaSuccess) return e;
  // ---- C: combine split partials
  if (h.balanced && h.grid > 1) {  // one block per CTA boundary and 16-row slice
    if (h.dh == 128)
      e = launch_c<128>(ap, h.grid - 1, stream);
    else
      e = launch_c<64>(ap, h.grid - 1, stream);
  }
  return e;
}

}  // namespace dflash

#ifdef DFLASH_WAIT_TEST
// Test build only: makes the producer of CTA `cta` skip the copy of its `tile`-th V tile
// (counted from 0 over the CTA's whole pass) in the following attention calls; cta = -1
// turns it off. Returns a cudaError_t.
extern "C" __attribute__((visibility("default"))) int dflash_test_withhold_v_tile(int cta, int tile) {
  const int2 v = make_int2(cta, tile);
  return static_cast<int>(cudaMemcpyToSymbol(dflash::g_withhold_v, &v, sizeof v));
}
#endif
