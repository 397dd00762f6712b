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
// lanes. The rotation angle of each lane's 8 frequencies is computed once per token.
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

template <int DH>
__device__ __forceinline__ void norm_rope_rows(const NormRopeJob& job, int64_t warp_id, int64_t n_warps) {
  constexpr int LR = DH / 8;       // lanes per row
  constexpr int HL = LR / 2;       // lanes per half row
  constexpr int RPS = 32 / LR;     // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane % LR;
  const int half = sub / HL;
  const int q = sub % HL;
  const int elem0 = half * (DH / 2) + 8 * q;
  const int pelem0 = (1 - half) * (DH / 2) + 8 * q;  // partner's elements
  const int row_in_step = lane / LR;
  const float sgn = half ? 1.0f : -1.0f;

  // weights of this lane's and the partner's elements, per part
  float w_me[2][8], w_pa[2][8];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (p < job.nparts) {
      const uint4 a = *reinterpret_cast<const uint4*>(job.part[p].w + elem0);
      const uint4 b = *reinterpret_cast<const uint4*>(job.part[p].w + pelem0);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        w_me[p][2 * e] = bf16lo_to_f32(av[e]);
        w_me[p][2 * e + 1] = bf16hi_to_f32(av[e]);
        w_pa[p][2 * e] = bf16lo_to_f32(bv[e]);
        w_pa[p][2 * e + 1] = bf16hi_to_f32(bv[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) w_me[p][e] = w_pa[p][e] = 0.0f;
    }
  }
  float thi[8], tlo[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    thi[e] = job.turns.hi[8 * q + e];
    tlo[e] = job.turns.lo[8 * q + e];
  }
  const float inv_dh = 1.0f / static_cast<float>(DH);

  for (int64_t t = warp_id; t < job.n_tok; t += n_warps) {
    int64_t dst_row = t;
    if (job.slot) {
      const int32_t s = job.slot[t];
      if (s < 0 || s >= job.capacity) {
        if (lane == 0 && job.err) atomicOr(job.err, kErrMetadata);
        continue;
      }
      dst_row = s;
    }
    const int pos = job.pos[t];
    float c[8], s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sincospif(2.0f * rope_turns(pos, thi[e], tlo[e]), &s[e], &c[e]);

#pragma unroll
    for (int p = 0; p < 2; ++p) {
      if (p >= job.nparts) break;
      const NormRopePart& P = job.part[p];
      for (int h0 = 0; h0 < P.heads; h0 += RPS) {
        const int h = h0 + row_in_step;
        const bool active = h < P.heads;
        const int64_t src_off = (t * P.heads + (active ? h : 0)) * DH;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (active) raw = *reinterpret_cast<const uint4*>(P.src + src_off + elem0);
        float x[8];
        {
          const uint32_t rv[4] = {raw.x, raw.y, raw.z, raw.w};
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
        uint4 praw;
        praw.x = __shfl_xor_sync(0xffffffffu, raw.x, HL);
        praw.y = __shfl_xor_sync(0xffffffffu, raw.y, HL);
        praw.z = __shfl_xor_sync(0xffffffffu, raw.z, HL);
        praw.w = __shfl_xor_sync(0xffffffffu, raw.w, HL);
        float xp[8];
        {
          const uint32_t rv[4] = {praw.x, praw.y, praw.z, praw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            xp[2 * e] = bf16lo_to_f32(rv[e]);
            xp[2 * e + 1] = bf16hi_to_f32(rv[e]);
          }
        }
        uint32_t ohi[4], olo[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float y0 = x[e] * rs * w_me[p][e], y1 = x[e + 1] * rs * w_me[p][e + 1];
          const float z0 = xp[e] * rs * w_pa[p][e], z1 = xp[e + 1] * rs * w_pa[p][e + 1];
          const float o0 = fmaf(sgn * z0, s[e], y0 * c[e]);
          const float o1 = fmaf(sgn * z1, s[e + 1], y1 * c[e + 1]);
          const uint32_t hi = pack_bf16x2(o0, o1);
          ohi[e / 2] = hi;
          olo[e / 2] = pack_bf16x2(o0 - bf16lo_to_f32(hi), o1 - bf16hi_to_f32(hi));
        }
        if (active) {
          const int64_t dst_off = (dst_row * P.heads + h) * DH + elem0;
          *reinterpret_cast<uint4*>(P.dst_hi + dst_off) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
          if (P.dst_lo) *reinterpret_cast<uint4*>(P.dst_lo + dst_off) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
          if (P.v_src) {
            const uint4 v = *reinterpret_cast<const uint4*>(P.v_src + src_off + elem0);
            *reinterpret_cast<uint4*>(P.v_dst + dst_off) = v;
          }
        }
      }
    }
  }
}

}  // namespace dflash
