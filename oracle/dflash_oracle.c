/*
 * dflash_oracle.c -- reference ("oracle") implementation of the DFlash draft
 * block-attention path, in plain C and IEEE double precision.
 *
 * TEST INFRASTRUCTURE. This is the slow, plainly written definition that the CUDA
 * path is checked against. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load it; the library itself never does. It shares no
 * code, header, table or constant with the CUDA sources.
 *
 * Source of each definition (vllm.cpp, a C++ port of vLLM):
 *   qwen3_dflash.cpp, PrecomputeContextKVDevice: context K gets the per-head k_norm
 *     (RMSNorm over head_dim) and then NeoX RoPE at the context positions; V is raw.
 *   qwen3_dflash.cpp, ForwardBlockLogits / ForwardWithCtxKVDev / ForwardPagedBody:
 *     block q and k get q_norm / k_norm (RmsNormArgs{eps, false}: the plain, non-gemma
 *     form) and then RopeNeox at the block positions; scale = 1/sqrt(head_dim).
 *   qwen3.cpp, file header: per-head q_norm/k_norm are applied BEFORE RoPE.
 *   qwen3_dflash.cpp, ForwardWithCtxKVDev: each request's attention runs over its
 *     combined sequence [context rows ; block rows] (cu_comb, ctx_dest, blk_idx), with
 *     DFlashBlockAttention's causal / sliding_window arguments; only block rows are kept
 *     (IndexSelect by blk_idx), as the paged variant computes them directly.
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   - RoPE: rotary dim = head_dim, inv_freq_i = theta^(-2i/Dh), pairs (i, i + Dh/2).
 *   - Mask, on combined indices i (query) and j (key) of one request:
 *       non-causal: every key of the request;  causal: j <= i;
 *       window W > 0 (only with causal): additionally i - j < W.
 *   - GQA: query head h reads kv head h / (Hq / Hkv).
 *
 * Tensor inputs are bfloat16 bit patterns (uint16), widened exactly to double.
 * Context keys passed to the attention functions are the stored (already normed and
 * rotated) keys, as the draft model stores them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

static double bf(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* RMSNorm of one head vector, plain (non-gemma) form:
 *   y_i = x_i / sqrt(mean_j(x_j^2) + eps) * w_i                                     */
static void rms_norm(const double* x, const double* w, int dh, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < dh; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / sqrt(ss / (double)dh + eps);
  for (int i = 0; i < dh; ++i) y[i] = x[i] * inv * w[i];
}

/* NeoX ("rotate half") rotary embedding at integer position pos, in place:
 *   for i < Dh/2, a = pos * theta^(-2i/Dh):
 *     y_i        = x_i cos a - x_{i+Dh/2} sin a
 *     y_{i+Dh/2} = x_{i+Dh/2} cos a + x_i sin a                                    */
static void rope_neox(double* y, int dh, double pos, double theta) {
  const int half = dh / 2;
  for (int i = 0; i < half; ++i) {
    const double a = pos * pow(theta, -2.0 * (double)i / (double)dh);
    const double c = cos(a), s = sin(a);
    const double x1 = y[i], x2 = y[i + half];
    y[i] = x1 * c - x2 * s;
    y[i + half] = x2 * c + x1 * s;
  }
}

static void load_row(const uint16_t* src, int dh, double* dst) {
  for (int i = 0; i < dh; ++i) dst[i] = bf(src[i]);
}

static void load_w(const uint16_t* w, int dh, double* dst) {
  for (int i = 0; i < dh; ++i) dst[i] = w ? bf(w[i]) : 1.0;
}

/* RMSNorm rows of x [n_tok, n_heads, dh] (bf16) into y (double); w == NULL means w = 1. */
int orc_rms_norm_rows(const uint16_t* x, const uint16_t* w, int64_t n_tok, int n_heads, int dh,
                      double eps, double* y) {
  if (n_tok < 0 || n_heads <= 0 || dh <= 0 || dh > 1024) return ORC_EINVAL;
  double wd[1024];
  load_w(w, dh, wd);
  const int64_t rows = n_tok * n_heads;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double xr[1024];
    load_row(x + r * dh, dh, xr);
    rms_norm(xr, wd, dh, eps, y + r * dh);
  }
  return ORC_OK;
}

/* NeoX RoPE on rows of x [n_tok, n_heads, dh] (double, any values) at pos[token]. */
int orc_rope_neox_rows(const double* x, const int32_t* pos, int64_t n_tok, int n_heads, int dh,
                       double theta, double* y) {
  if (n_tok < 0 || n_heads <= 0 || dh <= 0 || (dh & 1)) return ORC_EINVAL;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n_tok; ++t)
    for (int h = 0; h < n_heads; ++h) {
      const int64_t r = t * n_heads + h;
      memcpy(y + r * dh, x + r * dh, sizeof(double) * (size_t)dh);
      rope_neox(y + r * dh, dh, (double)pos[t], theta);
    }
  return ORC_OK;
}

/* One (token, head) row: RMSNorm with w, then NeoX RoPE at pos. */
static void norm_rope_row(const uint16_t* x, const double* w, int dh, double eps, double pos,
                          double theta, double* y) {
  double xr[1024];
  load_row(x, dh, xr);
  rms_norm(xr, w, dh, eps, y);
  rope_neox(y, dh, pos, theta);
}

/* Norm-then-rotate every row of x [n_tok, n_heads, dh]: the q/k prologue of the
 * block forward and, with the context positions, the context-K store. */
int orc_norm_rope(const uint16_t* x, const uint16_t* w, const int32_t* pos, int64_t n_tok,
                  int n_heads, int dh, double eps, double theta, double* y) {
  if (n_tok < 0 || n_heads <= 0 || dh <= 0 || dh > 1024 || (dh & 1)) return ORC_EINVAL;
  double wd[1024];
  load_w(w, dh, wd);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n_tok; ++t)
    for (int h = 0; h < n_heads; ++h) {
      const int64_t r = t * n_heads + h;
      norm_rope_row(x + r * dh, wd, dh, eps, (double)pos[t], theta, y + r * dh);
    }
  return ORC_OK;
}

/* Rounds a double to the nearest bfloat16 (ties to even) and returns its bits. The
 * draft model stores its context K/V as bf16 tensors, so a stored key is this value. */
static uint16_t to_bf16(double x) {
  if (x == 0.0 || !isfinite(x)) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
  }
  int e;
  const double m = frexp(x, &e);             /* x = m * 2^e, 0.5 <= |m| < 1 */
  const double r = ldexp(rint(ldexp(m, 8)), e - 8); /* keep 8 significant bits */
  float f = (float)r;                        /* exact: r has 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

int orc_round_bf16(const double* x, int64_t n, uint16_t* out) {
  if (n < 0) return ORC_EINVAL;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = to_bf16(x[i]);
  return ORC_OK;
}

/* Context-K store of the draft model: k_norm then RoPE at ctx_pos, V untouched.
 * out_f64 receives the exact values, out_bf16 (optional) the stored bf16 bits. */
int orc_context_kv(const uint16_t* k_raw, const int32_t* ctx_pos, const uint16_t* k_norm_w,
                   int64_t n_ctx, int hkv, int dh, double eps, double theta, double* out_f64,
                   uint16_t* out_bf16) {
  int rc = orc_norm_rope(k_raw, k_norm_w, ctx_pos, n_ctx, hkv, dh, eps, theta, out_f64);
  if (rc != ORC_OK) return rc;
  if (out_bf16) rc = orc_round_bf16(out_f64, n_ctx * hkv * dh, out_bf16);
  return rc;
}

typedef struct {
  const uint16_t *q, *k_blk, *v_blk, *ctx_k, *ctx_v, *q_norm_w, *k_norm_w;
  const int32_t *qsl, *csl, *clen, *positions;
  int n_req, hq, hkv, dh, causal, window;
  int64_t total_q, total_ctx;
  double eps, theta, scale;
} orc_args;

static int check_args(const orc_args* a) {
  if (a->n_req < 0 || a->hq <= 0 || a->hkv <= 0 || a->hq % a->hkv) return ORC_EINVAL;
  if (a->dh <= 0 || a->dh > 1024 || (a->dh & 1)) return ORC_EINVAL;
  if (a->window > 0 && !a->causal) return ORC_EINVAL;
  if (a->qsl[0] != 0 || a->qsl[a->n_req] != a->total_q) return ORC_EINVAL;
  for (int r = 0; r < a->n_req; ++r) {
    if (a->qsl[r + 1] < a->qsl[r] || a->csl[r + 1] < a->csl[r]) return ORC_EINVAL;
    if (a->clen[r] < 0 || a->clen[r] > a->csl[r + 1] - a->csl[r]) return ORC_EINVAL;
  }
  if (a->n_req > 0 && a->csl[a->n_req] > a->total_ctx) return ORC_EINVAL;
  return ORC_OK;
}

/* Mask of one request's combined sequence: query at combined index i, key at j. */
static int allowed(int64_t i, int64_t j, int causal, int window) {
  if (causal && j > i) return 0;
  if (window > 0 && i - j >= window) return 0;
  return 1;
}

/* Attention output of block row t (request r, block index b) for query head h.
 * Keys: the request's C_r context rows, then its B_r block rows (combined order).
 * Two passes: scores and their maximum, then exp-weights, their sum and the
 * weighted sum of V rows. */
static void attend_row(const orc_args* a, int r, int64_t t, int h, const double* wq,
                       const double* wk, double* out, double* scratch) {
  const int dh = a->dh, g = a->hq / a->hkv, kvh = h / g;
  const int64_t c = a->clen[r], b0 = a->qsl[r], nb = a->qsl[r + 1] - b0;
  const int64_t i = c + (t - b0); /* combined query index */
  double qh[1024], kh[1024];
  norm_rope_row(a->q + (t * a->hq + h) * dh, wq, dh, a->eps, (double)a->positions[t], a->theta, qh);
  double* s = scratch; /* [c + nb] scores */
  double m = -INFINITY;
  for (int64_t j = 0; j < c + nb; ++j) {
    if (!allowed(i, j, a->causal, a->window)) { s[j] = -INFINITY; continue; }
    const double* kp;
    if (j < c) {
      load_row(a->ctx_k + ((a->csl[r] + j) * a->hkv + kvh) * dh, dh, kh);
      kp = kh;
    } else {
      const int64_t tk = b0 + (j - c);
      norm_rope_row(a->k_blk + (tk * a->hkv + kvh) * dh, wk, dh, a->eps, (double)a->positions[tk],
                    a->theta, kh);
      kp = kh;
    }
    double dot = 0.0;
    for (int d = 0; d < dh; ++d) dot += qh[d] * kp[d];
    s[j] = a->scale * dot;
    if (s[j] > m) m = s[j];
  }
  for (int d = 0; d < dh; ++d) out[d] = 0.0;
  double l = 0.0;
  for (int64_t j = 0; j < c + nb; ++j) {
    if (s[j] == -INFINITY) continue;
    const double p = exp(s[j] - m);
    l += p;
    const uint16_t* vp = j < c ? a->ctx_v + ((a->csl[r] + j) * a->hkv + kvh) * dh
                               : a->v_blk + ((b0 + (j - c)) * a->hkv + kvh) * dh;
    for (int d = 0; d < dh; ++d) out[d] += p * bf(vp[d]);
  }
  for (int d = 0; d < dh; ++d) out[d] /= l;
}

static int request_of(const int32_t* qsl, int n_req, int64_t t) {
  int lo = 0, hi = n_req - 1;
  while (lo < hi) { /* last r with qsl[r] <= t and a non-empty block */
    const int mid = (lo + hi + 1) / 2;
    if (qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

static int run_rows(const orc_args* a, int64_t n_samples, const int32_t* sample_t,
                    const int32_t* sample_h, double* out) {
  int rc = check_args(a);
  if (rc != ORC_OK) return rc;
  double wq[1024], wk[1024];
  load_w(a->q_norm_w, a->dh, wq);
  load_w(a->k_norm_w, a->dh, wk);
  int64_t max_keys = 1;
  for (int r = 0; r < a->n_req; ++r) {
    const int64_t n = (int64_t)a->clen[r] + (a->qsl[r + 1] - a->qsl[r]);
    if (n > max_keys) max_keys = n;
  }
  int bad = 0;
#pragma omp parallel
  {
    double* scratch = (double*)malloc(sizeof(double) * (size_t)max_keys);
    if (!scratch) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t k = 0; k < n_samples; ++k) {
      if (!scratch) continue;
      const int64_t t = sample_t ? sample_t[k] : k / a->hq;
      const int h = sample_h ? sample_h[k] : (int)(k % a->hq);
      if (t < 0 || t >= a->total_q || h < 0 || h >= a->hq) {
#pragma omp atomic write
        bad = 2;
        continue;
      }
      attend_row(a, request_of(a->qsl, a->n_req, t), t, h, wq, wk, out + k * a->dh, scratch);
    }
    free(scratch);
  }
  return bad == 1 ? ORC_ENOMEM : bad == 2 ? ORC_EINVAL : ORC_OK;
}

#define ORC_ATTN_PARAMS                                                                      \
  const uint16_t *q, const uint16_t *k_blk, const uint16_t *v_blk, const uint16_t *ctx_k,    \
      const uint16_t *ctx_v, const int32_t *query_start_loc, const int32_t *ctx_start_loc,    \
      const int32_t *ctx_lens, const int32_t *positions, const uint16_t *q_norm_w,           \
      const uint16_t *k_norm_w, int n_req, int64_t total_q, int hq, int hkv, int dh,          \
      int64_t total_ctx, double eps, double theta, double scale, int causal, int window

#define ORC_FILL_ARGS(a)                                                                     \
  orc_args a = {q, k_blk, v_blk, ctx_k, ctx_v, q_norm_w, k_norm_w, query_start_loc,          \
                ctx_start_loc, ctx_lens, positions, n_req, hq, hkv, dh, causal, window,       \
                total_q, total_ctx, eps, theta, scale > 0.0 ? scale : 1.0 / sqrt((double)dh)}

/* Block attention for every block row and query head: out [total_q, hq, dh]. */
int orc_block_attention(ORC_ATTN_PARAMS, double* out) {
  ORC_FILL_ARGS(a);
  return run_rows(&a, total_q * hq, NULL, NULL, out);
}

/* The same, only for the listed (block row, query head) samples: out [n, dh]. */
int orc_block_attention_sampled(ORC_ATTN_PARAMS, int64_t n_samples, const int32_t* sample_t,
                                const int32_t* sample_h, double* out) {
  ORC_FILL_ARGS(a);
  return run_rows(&a, n_samples, sample_t, sample_h, out);
}

/* Brute force in the draft model's materialised form: build the combined
 * [context ; block] sequence of every request with the cu_comb / ctx_dest / blk_idx
 * maps, fill a dense score matrix for ALL combined rows (context query rows are zero,
 * as the combined q buffer is zeroed there), apply the mask matrix, take the row
 * softmax, multiply by V, and gather the block rows back by blk_idx. Small sizes only. */
int orc_block_attention_dense(ORC_ATTN_PARAMS, double* out) {
  ORC_FILL_ARGS(a);
  int rc = check_args(&a);
  if (rc != ORC_OK) return rc;
  const int g = hq / hkv;
  double wq[1024], wk[1024];
  load_w(q_norm_w, dh, wq);
  load_w(k_norm_w, dh, wk);
  /* combined layout */
  int64_t* cu_comb = (int64_t*)calloc((size_t)n_req + 1, sizeof(int64_t));
  if (!cu_comb) return ORC_ENOMEM;
  for (int r = 0; r < n_req; ++r)
    cu_comb[r + 1] = cu_comb[r] + ctx_lens[r] + (query_start_loc[r + 1] - query_start_loc[r]);
  const int64_t ncomb = cu_comb[n_req];
  int64_t* blk_idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total_q > 0 ? total_q : 1));
  double* qc = (double*)calloc((size_t)(ncomb * hq * dh) + 1, sizeof(double));
  double* kc = (double*)calloc((size_t)(ncomb * hkv * dh) + 1, sizeof(double));
  double* vc = (double*)calloc((size_t)(ncomb * hkv * dh) + 1, sizeof(double));
  double* oc = (double*)calloc((size_t)(ncomb * hq * dh) + 1, sizeof(double));
  if (!blk_idx || !qc || !kc || !vc || !oc) {
    free(cu_comb); free(blk_idx); free(qc); free(kc); free(vc); free(oc);
    return ORC_ENOMEM;
  }
  for (int r = 0; r < n_req; ++r) {
    const int64_t base = cu_comb[r];
    for (int64_t j = 0; j < ctx_lens[r]; ++j) /* ctx_dest: context row -> combined row */
      for (int h = 0; h < hkv; ++h)
        for (int d = 0; d < dh; ++d) {
          const int64_t src = ((ctx_start_loc[r] + j) * hkv + h) * dh + d;
          kc[((base + j) * hkv + h) * dh + d] = bf(ctx_k[src]);
          vc[((base + j) * hkv + h) * dh + d] = bf(ctx_v[src]);
        }
    const int64_t bbase = base + ctx_lens[r];
    for (int64_t t = query_start_loc[r]; t < query_start_loc[r + 1]; ++t) {
      const int64_t row = bbase + (t - query_start_loc[r]);
      blk_idx[t] = row;
      for (int h = 0; h < hq; ++h)
        norm_rope_row(q + (t * hq + h) * dh, wq, dh, eps, (double)positions[t], a.theta,
                      qc + (row * hq + h) * dh);
      for (int h = 0; h < hkv; ++h) {
        norm_rope_row(k_blk + (t * hkv + h) * dh, wk, dh, eps, (double)positions[t], a.theta,
                      kc + (row * hkv + h) * dh);
        for (int d = 0; d < dh; ++d) vc[(row * hkv + h) * dh + d] = bf(v_blk[(t * hkv + h) * dh + d]);
      }
    }
  }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int r = 0; r < n_req; ++r)
    for (int h = 0; h < hq; ++h) {
      const int64_t base = cu_comb[r], len = cu_comb[r + 1] - cu_comb[r];
      if (len == 0) continue;
      double* S = (double*)malloc(sizeof(double) * (size_t)(len * len));
      if (!S) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const int kvh = h / g;
      for (int64_t i = 0; i < len; ++i) {
        double m = -INFINITY;
        for (int64_t j = 0; j < len; ++j) {
          double dot = 0.0;
          for (int d = 0; d < dh; ++d)
            dot += qc[((base + i) * hq + h) * dh + d] * kc[((base + j) * hkv + kvh) * dh + d];
          S[i * len + j] = allowed(i, j, causal, window) ? a.scale * dot : -INFINITY;
          if (S[i * len + j] > m) m = S[i * len + j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < len; ++j) {
          S[i * len + j] = S[i * len + j] == -INFINITY ? 0.0 : exp(S[i * len + j] - m);
          l += S[i * len + j];
        }
        for (int64_t j = 0; j < len; ++j) S[i * len + j] /= l;
        for (int d = 0; d < dh; ++d) {
          double acc = 0.0;
          for (int64_t j = 0; j < len; ++j) acc += S[i * len + j] * vc[((base + j) * hkv + kvh) * dh + d];
          oc[((base + i) * hq + h) * dh + d] = acc;
        }
      }
      free(S);
    }
  if (!bad) /* IndexSelect of the block rows */
    for (int64_t t = 0; t < total_q; ++t)
      memcpy(out + t * hq * dh, oc + blk_idx[t] * hq * dh, sizeof(double) * (size_t)(hq * dh));
  free(cu_comb); free(blk_idx); free(qc); free(kc); free(vc); free(oc);
  return bad ? ORC_ENOMEM : ORC_OK;
}
