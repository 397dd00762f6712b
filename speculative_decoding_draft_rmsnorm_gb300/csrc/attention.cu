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
//      (bf16; in precise mode also the bf16 remainders), and, in block 0, the table of
//      work units: (request, kv head, query tile, range of key tiles).
//   B  attention: persistent CTAs, one per SM, walk their units round-robin.
//      Warp 0 streams Q / K / V tiles with TMA (128-byte swizzle); warp 1 issues
//      tcgen05 MMAs: S = Q K^T into tensor memory (M = 64 query rows = G heads x block
//      tokens, N = 128 keys), and O += P V (N = Dh) from P in shared memory; warps 2-5
//      run the online softmax (f32, base 2, lazy rescale of O in TMEM when the running
//      maximum grows by more than 2^8) and the epilogue. A unit covering all of a
//      request's keys writes the normalised output; a split unit writes (O, m, l).
//   C  combine: merges the split partials of a unit group:
//      o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
//
// TMEM map (512 columns): S[0] at column 0, S[1] at 128, O at 256. An M = 64 MMA puts
// query row rho in lane 32*(rho/16) + rho%16; softmax warp w (sub-partition w%4) owns
// rows 16*(w%4) .. +15, lanes 0-15 of the warp taking key columns 0-63 and lanes
// 16-31 columns 64-127 (tcgen05.ld 16x32bx2).
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
  Unit* units;
  uint32_t* hdr;
  int64_t total_q, total_ctx;
  int num_reqs, hkv, g, tpq, causal, window;
  int tiles_per_split, max_splits, units_max, max_ctx_len, max_block_len;
};

__device__ void build_units(const PrologueParams& p) {
  __shared__ int s_scan[256];
  __shared__ int s_bad_global;
  const int tid = threadIdx.x;
  if (tid == 0) {
    p.hdr[0] = 0;  // error word of this call (only this block writes it before kernel B)
    int bad = 0;
    if (p.num_reqs > 0 && (p.qsl[0] != 0 || p.qsl[p.num_reqs] != p.total_q)) bad = 1;
    s_bad_global = bad;
    if (bad) atomicOr(&p.hdr[0], kErrMetadata);
  }
  __syncthreads();
  const bool bad_global = s_bad_global != 0;
  int running = 0;
  for (int base = 0; base < p.num_reqs; base += 256) {
    const int r = base + tid;
    int cnt = 0, B = 0, C = 0, lo = 0, nct = 0, n = 0, QT = 0, S = 0, c0 = 0, q0 = 0;
    if (r < p.num_reqs && !bad_global) {
      q0 = p.qsl[r];
      const int q1 = p.qsl[r + 1];
      c0 = p.csl[r];
      const int c1 = p.csl[r + 1];
      B = q1 - q0;
      C = p.clen[r];
      const bool ok = B >= 0 && q0 >= 0 && q1 <= p.total_q && c0 >= 0 && c1 >= c0 && c1 <= p.total_ctx && C >= 0 &&
                      C <= c1 - c0 && C <= p.max_ctx_len && B <= p.max_block_len;
      if (!ok) {
        atomicOr(&p.hdr[0], kErrMetadata);
        B = 0;
      }
      if (B > 0) {
        lo = (p.causal && p.window > 0) ? max(0, C - p.window + 1) : 0;
        nct = (C - lo + kTileKeys - 1) / kTileKeys;
        n = nct + (B + kTileKeys - 1) / kTileKeys;
        QT = (B + p.tpq - 1) / p.tpq;
        S = (n + p.tiles_per_split - 1) / p.tiles_per_split;
        S = min(max(S, 1), min(p.max_splits, n));
        cnt = p.hkv * QT * S;
      }
    }
    // block-wide exclusive scan of cnt
    s_scan[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < 256; off <<= 1) {
      const int v = tid >= off ? s_scan[tid - off] : 0;
      __syncthreads();
      s_scan[tid] += v;
      __syncthreads();
    }
    const int offset = running + s_scan[tid] - cnt;
    const int chunk_total = s_scan[255];
    __syncthreads();
    if (cnt > 0) {
      for (int kvh = 0; kvh < p.hkv; ++kvh)
        for (int qt = 0; qt < QT; ++qt) {
          const int first = offset + (kvh * QT + qt) * S;
          for (int s = 0; s < S; ++s) {
            const int u = first + s;
            if (u >= p.units_max) {
              atomicOr(&p.hdr[0], kErrMetadata);
              continue;
            }
            Unit U;
            U.r = r;
            U.kvh = kvh;
            U.qt = qt;
            U.t0 = (s * n) / S;
            U.t1 = ((s + 1) * n) / S;
            U.split = s;
            U.nsplit = S;
            U.first = first;
            U.clen = C;
            U.blen = B;
            U.ctx_lo = lo;
            U.n_ctx_tiles = nct;
            U.csl = c0;
            U.qsl = q0;
            U.tok0 = qt * p.tpq;
            U.rows = min(p.tpq, B - U.tok0) * p.g;
            p.units[u] = U;
          }
        }
    }
    running += chunk_total;
  }
  if (tid == 0) p.hdr[1] = static_cast<uint32_t>(min(running, p.units_max));
}

template <int DH>
__global__ void __launch_bounds__(256) prologue_kernel(const __grid_constant__ PrologueParams p) {
  grid_dependents_launch();
  if (blockIdx.x == 0) {
    build_units(p);
    return;
  }
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x - 1) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x - 1) * blockDim.x) >> 5;
  norm_rope_rows<DH>(p.job, warp_id, n_warps);
}

// ================================================================ kernel B
template <int DH, int NK, int NV>
struct Layout {
  static constexpr int NB = DH / 64;                  // 128-byte column blocks per row
  static constexpr int QB = kTileRows * DH * 2;       // Q tile
  static constexpr int PB = kTileRows * kTileKeys * 2;  // P tile
  static constexpr int KB = kTileKeys * DH * 2;       // K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_P = OFF_Q + 2 * QB;
  static constexpr int OFF_K = OFF_P + 2 * PB;
  static constexpr int OFF_V = OFF_K + NK * KB;
  static constexpr int OFF_BAR = OFF_V + NV * KB;
  // barrier indices
  static constexpr int K_FULL = 0, K_EMPTY = NK, V_FULL = 2 * NK, V_EMPTY = 2 * NK + NV;
  static constexpr int Q_FULL = 2 * NK + 2 * NV, Q_EMPTY = Q_FULL + 2, S_FULL = Q_FULL + 4, S_EMPTY = Q_FULL + 6;
  static constexpr int P_FULL = Q_FULL + 8, P_EMPTY = Q_FULL + 10, O_FULL = Q_FULL + 12, O_EMPTY = Q_FULL + 13;
  static constexpr int DRAIN = Q_FULL + 14;  // final commit of the MMA thread (its own barrier)
  static constexpr int NBARS = Q_FULL + 15;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
};

struct AttnParams {
  const Unit* units;
  uint32_t* hdr;
  float* part_o;
  float* part_ml;
  void* out;
  int hq, g, out_f32, causal, window;
  float scale_log2;
};

struct TileInfo {
  int row;    // first source row (TMA outer coordinate)
  int valid;  // keys of this tile that belong to the request
  int j0;     // combined key index of the tile's first key
  bool blk;   // block-key tile (else context tile)
};

__device__ __forceinline__ TileInfo tile_info(const Unit& U, int t) {
  TileInfo ti;
  if (t < U.n_ctx_tiles) {
    const int k0 = U.ctx_lo + t * kTileKeys;
    ti.row = U.csl + k0;
    ti.valid = min(kTileKeys, U.clen - k0);
    ti.j0 = k0;
    ti.blk = false;
  } else {
    const int k0 = (t - U.n_ctx_tiles) * kTileKeys;
    ti.row = U.qsl + k0;
    ti.valid = min(kTileKeys, U.blen - k0);
    ti.j0 = U.clen + k0;
    ti.blk = true;
  }
  return ti;
}

__device__ __forceinline__ void load_unit(const Unit* units, int u, Unit& U) {
  const int4* src = reinterpret_cast<const int4*>(units + u);
  int4* dst = reinterpret_cast<int4*>(&U);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = src[i];
}

template <int DH, int NK, int NV>
__global__ void __launch_bounds__(192, 1)
attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                 const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kb,
                 const __grid_constant__ CUtensorMap tm_vb, const __grid_constant__ AttnParams p) {
  using L = Layout<DH, NK, NV>;
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
      mbar_init(bar(L::Q_EMPTY + i), 1);
      mbar_init(bar(L::S_FULL + i), 1);
      mbar_init(bar(L::S_EMPTY + i), 4);
      mbar_init(bar(L::P_FULL + i), 4);
      mbar_init(bar(L::P_EMPTY + i), 1);
    }
    mbar_init(bar(L::O_FULL), 1);
    mbar_init(bar(L::O_EMPTY), 4);
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
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();  // unit table and q^/k^ come from the prologue kernel
  grid_dependents_launch();
  const int n_units = static_cast<int>(p.hdr[1]);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t gk = 0, gv = 0;
      int iu = 0;
      bool ok = true;
      constexpr uint32_t q_box_bytes_per_row = 128;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++iu) {
        Unit U;
        load_unit(p.units, u, U);
        const int qb = iu & 1;
        if (!(ok = mbar_wait(bar(L::Q_EMPTY + qb), ((iu >> 1) & 1) ^ 1, abort_flag))) break;
        // the Q box is G x (64 / G) rows whatever this unit's row count
        const uint32_t q_rows = static_cast<uint32_t>(p.g * (kTileRows / p.g));
        mbar_arrive_expect_tx(bar(L::Q_FULL + qb), L::NB * q_rows * q_box_bytes_per_row);
#pragma unroll
        for (int nb = 0; nb < L::NB; ++nb)
          tma_load_4d(sbase + L::OFF_Q + qb * L::QB + nb * (kTileRows * 128), &tm_q, bar(L::Q_FULL + qb), nb * 64, 0,
                      U.kvh, U.qsl + U.tok0);
        const int n = U.t1 - U.t0;
        auto issue_k = [&](int t) -> bool {
          const int slot = static_cast<int>(gk % NK);
          if (!mbar_wait(bar(L::K_EMPTY + slot), ((gk / NK) & 1) ^ 1, abort_flag)) return false;
          const TileInfo ti = tile_info(U, t);
          mbar_arrive_expect_tx(bar(L::K_FULL + slot), L::KB);
          const void* map = ti.blk ? static_cast<const void*>(&tm_kb) : static_cast<const void*>(&tm_kc);
#pragma unroll
          for (int nb = 0; nb < L::NB; ++nb)
            tma_load_3d(sbase + L::OFF_K + slot * L::KB + nb * (kTileKeys * 128), map, bar(L::K_FULL + slot), nb * 64,
                        U.kvh, ti.row);
          ++gk;
          return true;
        };
        auto issue_v = [&](int t) -> bool {
          const int slot = static_cast<int>(gv % NV);
          if (!mbar_wait(bar(L::V_EMPTY + slot), ((gv / NV) & 1) ^ 1, abort_flag)) return false;
          const TileInfo ti = tile_info(U, t);
          mbar_arrive_expect_tx(bar(L::V_FULL + slot), L::KB);
          const void* map = ti.blk ? static_cast<const void*>(&tm_vb) : static_cast<const void*>(&tm_vc);
#pragma unroll
          for (int nb = 0; nb < L::NB; ++nb)
            tma_load_3d(sbase + L::OFF_V + slot * L::KB + nb * (kTileKeys * 128), map, bar(L::V_FULL + slot), nb * 64,
                        U.kvh, ti.row);
          ++gv;
          return true;
        };
        if (!(ok = issue_k(U.t0))) break;
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) ok = issue_k(U.t0 + j + 1);
          if (ok) ok = issue_v(U.t0 + j);
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
    if (lane == 0) {
      uint32_t gk = 0, gv = 0, gj = 0;
      int iu = 0;
      bool ok = true;
      const uint32_t idesc_pv = umma_idesc_bf16(kTileRows, DH, 0, 1);
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++iu) {
        Unit U;
        load_unit(p.units, u, U);
        const int qb = iu & 1;
        const int n = U.t1 - U.t0;
        if (!(ok = mbar_wait(bar(L::Q_FULL + qb), (iu >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t q_addr = sbase + L::OFF_Q + qb * L::QB;
        auto issue_qk = [&](int j) -> bool {
          const uint32_t g = gj + j;
          const int sb = g & 1;
          const int slot = static_cast<int>(gk % NK);
          if (!mbar_wait(bar(L::K_FULL + slot), (gk / NK) & 1, abort_flag)) return false;
          if (!mbar_wait(bar(L::S_EMPTY + sb), ((g >> 1) & 1) ^ 1, abort_flag)) return false;
          tc_fence_after();
          const TileInfo ti = tile_info(U, U.t0 + j);
          const int nq = min(kTileKeys, (ti.valid + 15) & ~15);
          const uint32_t idesc = umma_idesc_bf16(kTileRows, nq, 0, 0);
          const uint32_t k_addr = sbase + L::OFF_K + slot * L::KB;
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint64_t a = umma_desc_sw128(q_addr + (kk >> 2) * (kTileRows * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t b = umma_desc_sw128(k_addr + (kk >> 2) * (kTileKeys * 128) + (kk & 3) * 32, 16, 1024);
            umma_bf16_ss(tmem + sb * 128, a, b, idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(L::S_FULL + sb));
          umma_commit(bar(L::K_EMPTY + slot));
          if (j == n - 1) umma_commit(bar(L::Q_EMPTY + qb));
          ++gk;
          return true;
        };
        if (!(ok = issue_qk(0))) break;
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n && !(ok = issue_qk(j + 1))) break;
          const uint32_t g = gj + j;
          const int pb = g & 1;
          const int vslot = static_cast<int>(gv % NV);
          if (!(ok = mbar_wait(bar(L::P_FULL + pb), (g >> 1) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(bar(L::V_FULL + vslot), (gv / NV) & 1, abort_flag))) break;
          if (j == 0 && !(ok = mbar_wait(bar(L::O_EMPTY), (iu & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          const TileInfo ti = tile_info(U, U.t0 + j);
          const int ksteps = (ti.valid + 15) >> 4;
          const uint32_t p_addr = sbase + L::OFF_P + pb * L::PB;
          const uint32_t v_addr = sbase + L::OFF_V + vslot * L::KB;
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint64_t a = umma_desc_sw128(p_addr + (kk >> 2) * (kTileRows * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t b = umma_desc_sw128(v_addr + kk * (16 * 128), kTileKeys * 128, 1024);
            umma_bf16_ss(tmem + 256, a, b, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(bar(L::V_EMPTY + vslot));
          umma_commit(bar(L::P_EMPTY + pb));
          ++gv;
        }
        if (!ok) break;
        umma_commit(bar(L::O_FULL));
        gj += n;
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
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++iu) {
      Unit U;
      load_unit(p.units, u, U);
      const int n = U.t1 - U.t0;
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
      for (int j = 0; j < n; ++j) {
        const uint32_t g = gj + j;
        const int sb = g & 1;
        const TileInfo ti = tile_info(U, U.t0 + j);
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
        float mt = -INFINITY;
        float x[64];
        if (full_tile) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            x[c] = __uint_as_float(sr[c]) * sl2;
            mt = fmaxf(mt, x[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int jj = jbase + c;
            const bool keep = (col0 + c < ti.valid) && jj >= jlo && jj <= jhi;
            x[c] = keep ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
            mt = fmaxf(mt, x[c]);
          }
        }
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
          constexpr int CH = DH / 2 / 32;  // 32-column chunks per half row of O
#pragma unroll
          for (int ch = 0; ch < CH; ++ch) {
            uint32_t o[32];
            tmem_ld_16x32bx2_x32<DH / 2>(tmem + lane_base + 256 + ch * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_16x32bx2_x32<DH / 2>(tmem + lane_base + 256 + ch * 32, o);
          }
          tmem_wait_st();
        }
        const float m_eff = m_used == -INFINITY ? 0.0f : m_used;
        uint32_t pk[32];
        float lsum = 0.0f;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = ex2_approx(x[c] - m_eff);
          const float p1 = ex2_approx(x[c + 1] - m_eff);
          const uint32_t v = pack_bf16x2(p0, p1);
          pk[c / 2] = v;
          lsum += bf16lo_to_f32(v) + bf16hi_to_f32(v);
        }
        l += lsum;
        // the P buffer is free once PV of tile g-2 has completed
        if (!(ok = wait_warp(bar(L::P_EMPTY + sb), ((g >> 1) & 1) ^ 1))) break;
        {
          uint8_t* prow = smem + L::OFF_P + sb * L::PB + half * (kTileRows * 128) + rho * 128;
#pragma unroll
          for (int chn = 0; chn < 8; ++chn) {
            uint4 v = make_uint4(pk[4 * chn], pk[4 * chn + 1], pk[4 * chn + 2], pk[4 * chn + 3]);
            *reinterpret_cast<uint4*>(prow + ((chn ^ (rho & 7)) << 4)) = v;
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
            *reinterpret_cast<uint4*>(smem + L::OFF_V + vslot * L::KB + nb * (kTileKeys * 128) + row * 128 + chn * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::P_FULL + sb));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = wait_warp(bar(L::O_FULL), iu & 1))) break;
      tc_fence_after();
      constexpr int CH = DH / 2 / 32;
      uint32_t o[CH][32];
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) tmem_ld_16x32bx2_x32<DH / 2>(tmem + lane_base + 256 + ch * 32, o[ch]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::O_EMPTY));
      const float l_tot = l + __shfl_xor_sync(0xffffffffu, l, 16);
      if (row_ok) {
        const int gi = rho % p.g;
        const int64_t tok = U.qsl + b;
        const int head = U.kvh * p.g + gi;
        if (U.nsplit == 1) {
          const float inv = l_tot > 0.0f ? 1.0f / l_tot : 0.0f;
          if (p.out_f32) {
            float* dst = reinterpret_cast<float*>(p.out) + (tok * p.hq + head) * DH + half * (DH / 2);
#pragma unroll
            for (int ch = 0; ch < CH; ++ch)
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(dst + ch * 32 + e) =
                    make_float4(__uint_as_float(o[ch][e]) * inv, __uint_as_float(o[ch][e + 1]) * inv,
                                __uint_as_float(o[ch][e + 2]) * inv, __uint_as_float(o[ch][e + 3]) * inv);
          } else {
            uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + (tok * p.hq + head) * DH + half * (DH / 2);
#pragma unroll
            for (int ch = 0; ch < CH; ++ch)
#pragma unroll
              for (int e = 0; e < 32; e += 8) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[ch][e]) * inv, __uint_as_float(o[ch][e + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(o[ch][e + 2]) * inv, __uint_as_float(o[ch][e + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(o[ch][e + 4]) * inv, __uint_as_float(o[ch][e + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(o[ch][e + 6]) * inv, __uint_as_float(o[ch][e + 7]) * inv);
                *reinterpret_cast<uint4*>(dst + ch * 32 + e) = v;
              }
          }
        } else {
          float* dst = p.part_o + (static_cast<int64_t>(u) * kTileRows + rho) * DH + half * (DH / 2);
#pragma unroll
          for (int ch = 0; ch < CH; ++ch)
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + ch * 32 + e) =
                  make_float4(__uint_as_float(o[ch][e]), __uint_as_float(o[ch][e + 1]), __uint_as_float(o[ch][e + 2]),
                              __uint_as_float(o[ch][e + 3]));
          if (half == 0) {
            float* ml = p.part_ml + (static_cast<int64_t>(u) * kTileRows + rho) * 2;
            ml[0] = m_used;
            ml[1] = l_tot;
          }
        }
      }
      gj += n;
      gv += n;
    }
    if (!ok) atomicOr(&p.hdr[0], kErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================ kernel C
template <int DH>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnParams p) {
  grid_dependency_wait();
  const int u = blockIdx.x;
  const int n_units = static_cast<int>(p.hdr[1]);
  if (u >= n_units) return;
  Unit U;
  load_unit(p.units, u, U);
  if (U.split != 0 || U.nsplit <= 1) return;
  if (u + U.nsplit > n_units) {  // group cut short by a truncated unit table
    if (threadIdx.x == 0) atomicOr(&p.hdr[0], kErrMetadata);
    return;
  }
  constexpr int CPR = DH / 8;  // 8-float chunks per row
  for (int item = threadIdx.x; item < U.rows * CPR; item += blockDim.x) {
    const int rho = item / CPR;
    const int c8 = (item % CPR) * 8;
    float M = -INFINITY;
    for (int s = 0; s < U.nsplit; ++s) M = fmaxf(M, p.part_ml[(static_cast<int64_t>(u + s) * kTileRows + rho) * 2]);
    const float Me = M == -INFINITY ? 0.0f : M;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float L = 0.0f;
    for (int s = 0; s < U.nsplit; ++s) {
      const float* ml = p.part_ml + (static_cast<int64_t>(u + s) * kTileRows + rho) * 2;
      const float w = ml[0] == -INFINITY ? 0.0f : ex2_approx(ml[0] - Me);
      L += w * ml[1];
      const float4* src = reinterpret_cast<const float4*>(p.part_o + (static_cast<int64_t>(u + s) * kTileRows + rho) * DH + c8);
      const float4 a = src[0], b = src[1];
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    const int64_t tok = U.qsl + U.tok0 + rho / p.g;
    const int head = U.kvh * p.g + rho % p.g;
    if (p.out_f32) {
      float* dst = reinterpret_cast<float*>(p.out) + (tok * p.hq + head) * DH + c8;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
    } else {
      uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + (tok * p.hq + head) * DH + c8;
      uint4 v;
      v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(dst) = v;
    }
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
  if (causal && window > 0) ctx_tiles_max = std::min(ctx_tiles_max, (window - 1 + kTileKeys - 1) / kTileKeys);
  const int blk_tiles_max = (max_block_len + kTileKeys - 1) / kTileKeys;
  const int n_max = std::max(1, ctx_tiles_max + blk_tiles_max);
  // tiles over all requests (per kv head and query tile), an upper bound from capacities
  double tiles_bound = static_cast<double>(total_ctx) / kTileKeys + static_cast<double>(num_reqs) * (1 + blk_tiles_max);
  if (causal && window > 0)
    tiles_bound = std::min(tiles_bound, static_cast<double>(num_reqs) * n_max);
  // aim for about two units per SM (tunable with DFLASH_TILES_PER_SPLIT)
  const double est = static_cast<double>(hkv) * std::max(1, w.qt_max) * tiles_bound;
  int tps = static_cast<int>(std::ceil(est / std::max(1, 2 * num_sms)));
  tps = std::max(tps, 4);
  if (const char* e = std::getenv("DFLASH_TILES_PER_SPLIT")) {
    const int v = std::atoi(e);
    if (v > 0) tps = v;
  }
  if (flags & 2) tps = n_max;                                   // DFLASH_FLAG_NO_SPLIT
  if (flags & 1) tps = std::min(tps, std::max(1, (n_max + 1) / 2));  // DFLASH_FLAG_FORCE_SPLIT
  w.tiles_per_split = tps;
  w.max_splits = std::max(1, (n_max + tps - 1) / tps);
  w.may_split = w.max_splits > 1;
  const double sum_splits = std::min(tiles_bound / tps + num_reqs, static_cast<double>(num_reqs) * w.max_splits);
  const double units = static_cast<double>(hkv) * std::max(1, w.qt_max) * sum_splits;
  w.units_max = static_cast<int>(std::min(units + 1.0, 2.0e9 / 64.0));
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
  w.units = off;
  off += align256(static_cast<size_t>(w.units_max) * sizeof(Unit));
  w.part_o = off;
  if (w.may_split) off += align256(static_cast<size_t>(w.units_max) * kTileRows * dh * 4);
  w.part_ml = off;
  if (w.may_split) off += align256(static_cast<size_t>(w.units_max) * kTileRows * 2 * 4);
  w.total = off;
  return w;
}

template <int DH, int NK, int NV>
static cudaError_t launch_b(const CUtensorMap& tq, const CUtensorMap& tkc, const CUtensorMap& tvc,
                            const CUtensorMap& tkb, const CUtensorMap& tvb, const AttnParams& ap, int grid,
                            cudaStream_t stream) {
  using L = Layout<DH, NK, NV>;
  static_assert(L::ALLOC <= 232448, "shared memory plan exceeds the per-block limit");
  auto kern = attention_kernel<DH, NK, NV>;
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
  return cudaLaunchKernelEx(&cfg, kern, tq, tkc, tvc, tkb, tvb, ap);
}

template <int DH>
static cudaError_t launch_c(const AttnParams& ap, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
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
  pp.units = h.units;
  pp.hdr = h.ws_hdr;
  pp.total_q = h.total_q;
  pp.total_ctx = h.total_ctx;
  pp.num_reqs = h.num_reqs;
  pp.hkv = h.hkv;
  pp.g = h.g;
  pp.tpq = h.tpq;
  pp.causal = h.causal;
  pp.window = h.window;
  pp.tiles_per_split = h.tiles_per_split;
  pp.max_splits = h.max_splits;
  pp.units_max = h.units_max;
  pp.max_ctx_len = h.max_ctx_len;
  pp.max_block_len = h.max_block_len;
  cudaError_t e = cudaSuccess;
  int64_t nr_blocks = (h.total_q + 7) / 8;
  nr_blocks = std::min<int64_t>(nr_blocks, static_cast<int64_t>(h.num_sms) * 2);  // all co-resident
  const unsigned grid_a = static_cast<unsigned>(1 + nr_blocks);
  if (h.dh == 128)
    prologue_kernel<128><<<grid_a, 256, 0, stream>>>(pp);
  else
    prologue_kernel<64><<<grid_a, 256, 0, stream>>>(pp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // ---- tensor maps
  CUtensorMap tq, tkc, tvc, tkb, tvb;
  const void* ctx_k = h.total_ctx > 0 ? static_cast<const void*>(h.ctx_k) : static_cast<const void*>(h.q_hat);
  const void* ctx_v = h.total_ctx > 0 ? static_cast<const void*>(h.ctx_v) : static_cast<const void*>(h.q_hat);
  const int64_t ctx_rows = h.total_ctx > 0 ? h.total_ctx : 1;
  bool ok = encode_q_map(&tq, h.q_hat, h.dh, h.g, h.hkv, h.total_q, h.tpq) &&
            encode_rows_map(&tkc, ctx_k, h.dh, h.hkv, ctx_rows, kTileKeys) &&
            encode_rows_map(&tvc, ctx_v, h.dh, h.hkv, ctx_rows, kTileKeys) &&
            encode_rows_map(&tkb, h.k_hat, h.dh, h.hkv, h.total_q, kTileKeys) &&
            encode_rows_map(&tvb, h.v_blk, h.dh, h.hkv, h.total_q, kTileKeys);
  if (!ok) {
    std::snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (driver entry point or tensor layout)");
    return cudaErrorInvalidValue;
  }
  AttnParams ap{};
  ap.units = h.units;
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
  const int grid_b = std::max(1, std::min(h.num_sms, h.units_max));
  // ---- B: attention
  if (h.dh == 128)
    e = launch_b<128, 3, 2>(tq, tkc, tvc, tkb, tvb, ap, grid_b, stream);
  else
    e = launch_b<64, 4, 4>(tq, tkc, tvc, tkb, tvb, ap, grid_b, stream);
  if (e != cudaSuccess) return e;
  // ---- C: combine split partials
  if (h.may_split) {
    if (h.dh == 128)
      e = launch_c<128>(ap, h.units_max, stream);
    else
      e = launch_c<64>(ap, h.units_max, stream);
  }
  return e;
}

}  // namespace dflash
