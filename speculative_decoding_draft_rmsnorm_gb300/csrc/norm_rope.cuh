// norm_rope.cuh -- fused per-head RMSNorm + NeoX RoPE (and the context-store write).
//
// Computes, per (token, head) row x of head_dim Dh (vllm.cpp qwen3_dflash.cpp:
// q_norm / k_norm with RmsNormArgs{eps, false}, then RopeNeox at the token position):
//     y = x / sqrt(mean(x^2) + eps) * w
//     for i < Dh/2, a = pos * theta^(-2i/Dh):
//        out_i        = y_i cos a - y_{i+Dh/2} sin a
//        out_{i+Dh/2} = y_{i+Dh/2} cos a + y_i sin a
// in f32, rounding once to bf16 (and optionally storing the bf16 remainder, so that
// hi + lo carries the f32 result to ~16 significant bits).
//
// Layout: one warp per token, all heads of the token. A row is covered by Dh/8 lanes
// holding 8 consecutive elements each (one 16-byte load): lanes of the first half hold
// elements [8q, 8q+8), lanes of the second half the partner elements [Dh/2 + 8q, ...),
// so the rotation partner of a lane is lane ^ (Dh/16). 32 / (Dh/8) rows are processed
// per warp step; the squared-norm reduction is a shuffle butterfly within the row's
// lanes. All rows of a warp's item belong to one token, so each of the Dh/2 rotation
// angles is computed by one lane (Dh/64 per lane) and fetched by the others with shuffles.
//
// Angle: turns = pos * (inv_freq / 2pi) is formed exactly with an FMA two-product of
// a float head/tail split of inv_freq/2pi (host-computed in double), reduced modulo 1
// exactly, and passed to sincospif; the result is accurate to a few 1e-7 rad at any
// position below 2^24, where a plain f32 product pos * inv_freq would be off by up to
// ~2e-3 rad at position 32k.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace dflash {

// pos * (hi + lo) modulo 1, in [-0.5, 0.5].
__device__ __forceinline__ float rope_turns(int pos, float hi, float lo) {
  const float ph = static_cast<float>(pos & ~4095);  // exact: at most 20 significant bits
  const float pl = static_cast<float>(pos & 4095);   // exact
  const float p1 = ph * hi, e1 = fmaf(ph, hi, -p1);  // p1 + e1 == ph * hi exactly
  const float p2 = pl * hi, e2 = fmaf(pl, hi, -p2);
  const float f1 = p1 - rintf(p1), f2 = p2 - rintf(p2);  // exact
  float t = (f1 + f2) + ((e1 + e2) + static_cast<float>(pos) * lo);
  return t - rintf(t);
}

// Whether request r's whole append fits: positions [L, L + count) with L = seq_lens[r] all
// fall inside its block table on page ids inside the pool. The page checks its store's
// capacity before it writes any row (qwen3_dflash.cpp, AppendContextKVDevice), so a request
// that does not fit writes nothing and keeps its length. `lane` / `lanes` split the page
// checks over the lanes of a warp (lanes = 32, every lane calls with its own lane; the
// result is the same on all of them) or run them in one thread (lane = 0, lanes = 1).
__device__ __forceinline__ bool append_fits(const AppendMap& m, int r, int lane, int lanes) {
  const int64_t L = m.seq_lens[r];
  const int64_t count = static_cast<int64_t>(m.new_start_loc[r + 1]) - m.new_start_loc[r];
  if (count <= 0) return true;
  const int64_t last = L + count - 1;
  if (L < 0 || last > 0x7fffffff || last / m.page_size >= m.max_pages) return false;
  bool ok = true;
  const int64_t p0 = L / m.page_size, p1 = last / m.page_size;
  const int32_t* row = m.block_table + static_cast<int64_t>(r) * m.max_pages;
  for (int64_t pg = p0 + lane; pg <= p1; pg += lanes) {
    const int id = row[pg];
    if (id < 0 || id >= m.num_pages) ok = false;
  }
  if (lanes > 1) ok = __all_sync(0xffffffffu, ok);
  return ok;
}

// Row t of a paged append (called by all lanes of a warp with the same t): 1 = mapped to
// (pos, dst); 0 = in no request (ignored); -1 = its request's append does not fit (reported,
// none of the request's rows is written).
__device__ __forceinline__ int append_row(const AppendMap& m, int64_t t, int* pos, int64_t* dst) {
  int lo = 0, hi = m.num_reqs + 1;  // first i with new_start_loc[i] > t
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (m.new_start_loc[mid] <= t) lo = mid + 1; else hi = mid;
  }
  const int r = lo - 1;
  if (r < 0 || r >= m.num_reqs) return 0;
  if (!append_fits(m, r, threadIdx.x & 31, 32)) return -1;
  const int64_t p = static_cast<int64_t>(m.seq_lens[r]) + (t - m.new_start_loc[r]);
  const int page = m.block_table[static_cast<int64_t>(r) * m.max_pages + p / m.page_size];
  *pos = static_cast<int>(p);
  *dst = static_cast<int64_t>(page) * m.page_size + p % m.page_size;
  return 1;
}

// Work item: one token and a chunk of up to RPS * kUnroll of its heads in one part. The
// chunk's loads (and V loads) are all issued before any arithmetic, so a warp keeps
// kUnroll 16-byte loads per lane in flight; items are spread over all warps of the grid.
// HAS_V = false drops the optional V copy (and its registers). APPEND takes each row's
// position and destination from *app instead of job.pos / job.slot.
template <int DH, bool HAS_V = true, bool APPEND = false>
__device__ __forceinline__ void norm_rope_rows(const NormRopeJob& job, int64_t warp_id, int64_t n_warps,
                                               const AppendMap* app = nullptr) {
  constexpr int LR = DH / 8;       // lanes per row
  constexpr int HL = LR / 2;       // lanes per half row
  constexpr int RPS = 32 / LR;     // rows per warp step
  constexpr int kUnroll = 4;       // warp steps per item
  constexpr int HPI = RPS * kUnroll;  // heads per item
  const int lane = threadIdx.x & 31;
  const int sub = lane % LR;
  const int half = sub / HL;
  const int q = sub % HL;
  const int elem0 = half * (DH / 2) + 8 * q;
  const int pelem0 = (1 - half) * (DH / 2) + 8 * q;  // partner's elements
  const int row_in_step = lane / LR;
  const float sgn = half ? 1.0f : -1.0f;
  const float inv_dh = 1.0f / static_cast<float>(DH);
  static_assert(DH == 64 || DH == 128, "head_dim 64 or 128");
  constexpr int FPL = DH / 64;  // frequencies computed per lane
  float thi[FPL], tlo[FPL];
#pragma unroll
  for (int i = 0; i < FPL; ++i) {
    thi[i] = job.turns.hi[lane * FPL + i];
    tlo[i] = job.turns.lo[lane * FPL + i];
  }
  const int chunks0 = (job.part[0].heads + HPI - 1) / HPI;
  const int chunks1 = job.nparts > 1 ? (job.part[1].heads + HPI - 1) / HPI : 0;
  const int cpt = chunks0 + chunks1;  // items per token
  const int64_t n_items = job.n_tok * cpt;

  for (int64_t item = warp_id; item < n_items; item += n_warps) {
    const int64_t t = item / cpt;
    const int c = static_cast<int>(item - t * cpt);
    const int p = c < chunks0 ? 0 : 1;
    const NormRopePart& P = job.part[p];
    const int hc = (p == 0 ? c : c - chunks0) * HPI;
    // issue every load of the item first
    uint4 raw[kUnroll], vraw[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int h = hc + u * RPS + row_in_step;
      raw[u] = make_uint4(0, 0, 0, 0);
      vraw[u] = make_uint4(0, 0, 0, 0);
      if (h < P.heads) {
        raw[u] = *reinterpret_cast<const uint4*>(P.src + (t * P.heads + h) * DH + elem0);
        if (HAS_V && P.v_src) vraw[u] = *reinterpret_cast<const uint4*>(P.v_src + (t * P.heads + h) * DH + elem0);
      }
    }
    // the row's destination (and, appending, its position) while its loads are in flight
    int64_t dst_row = t;
    int pos = 0;
    if constexpr (APPEND) {
      const int m = append_row(*app, t, &pos, &dst_row);
      if (m <= 0) {
        if (m < 0 && lane == 0 && job.err) atomicOr(job.err, kErrMetadata);
        continue;
      }
    } else if (job.slot) {
      const int32_t sl = job.slot[t];
      if (sl < 0 || sl >= job.capacity) {
        if (lane == 0 && job.err) atomicOr(job.err, kErrMetadata);
        continue;
      }
      dst_row = sl;
    }
    float w_me[8], w_pa[8];
    {
      const uint4 a = *reinterpret_cast<const uint4*>(P.w + elem0);
      const uint4 b = *reinterpret_cast<const uint4*>(P.w + pelem0);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        w_me[2 * e] = bf16lo_to_f32(av[e]);
        w_me[2 * e + 1] = bf16hi_to_f32(av[e]);
        w_pa[2 * e] = bf16lo_to_f32(bv[e]);
        w_pa[2 * e + 1] = bf16hi_to_f32(bv[e]);
      }
    }
    if constexpr (!APPEND) pos = job.pos[t];
    float mc[FPL], ms[FPL];  // this lane's frequencies lane * FPL + i
#pragma unroll
    for (int i = 0; i < FPL; ++i) sincospif(2.0f * rope_turns(pos, thi[i], tlo[i]), &ms[i], &mc[i]);
    float cs[8], sn[8];  // frequencies 8q + e, from lane (8q + e) / FPL (8q is a multiple of FPL)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int src = (8 * q + e) / FPL;
      cs[e] = __shfl_sync(0xffffffffu, mc[e % FPL], src);
      sn[e] = __shfl_sync(0xffffffffu, ms[e % FPL], src);
    }

#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int h = hc + u * RPS + row_in_step;
      float x[8], xp[8];
      {
        const uint32_t rv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[2 * e] = bf16lo_to_f32(rv[e]);
          x[2 * e + 1] = bf16hi_to_f32(rv[e]);
        }
      }
      float ss = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int o = 1; o < LR; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rs = rsqrtf(fmaf(ss, inv_dh, job.eps));
      {
        const uint32_t rv[4] = {__shfl_xor_sync(0xffffffffu, raw[u].x, HL), __shfl_xor_sync(0xffffffffu, raw[u].y, HL),
                                __shfl_xor_sync(0xffffffffu, raw[u].z, HL), __shfl_xor_sync(0xffffffffu, raw[u].w, HL)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xp[2 * e] = bf16lo_to_f32(rv[e]);
          xp[2 * e + 1] = bf16hi_to_f32(rv[e]);
        }
      }
      uint32_t ohi[4], olo[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float y0 = x[e] * rs * w_me[e], y1 = x[e + 1] * rs * w_me[e + 1];
        const float z0 = xp[e] * rs * w_pa[e], z1 = xp[e + 1] * rs * w_pa[e + 1];
        const float o0 = fmaf(sgn * z0, sn[e], y0 * cs[e]);
        const float o1 = fmaf(sgn * z1, sn[e + 1], y1 * cs[e + 1]);
        const uint32_t hi = pack_bf16x2(o0, o1);
        ohi[e / 2] = hi;
        olo[e / 2] = pack_bf16x2(o0 - bf16lo_to_f32(hi), o1 - bf16hi_to_f32(hi));
      }
      if (h < P.heads) {
        const int64_t dst_off = (dst_row * P.heads + h) * DH + elem0;
        *reinterpret_cast<uint4*>(P.dst_hi + dst_off) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
        if (P.dst_lo) *reinterpret_cast<uint4*>(P.dst_lo + dst_off) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
        if (HAS_V && P.v_src) *reinterpret_cast<uint4*>(P.v_dst + dst_off) = vraw[u];
      }
    }
  }
}

}  // namespace dflash
