/* CPU oracle for the fused MoE expert block (test infrastructure only).
 *
 * This file is the independent reference that the CUDA path is checked
 * against.  Only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg may load it; the product path never does.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * It follows the FusedDeepMoE analysis ("FusedDeepMoE Kernel 深度分析报告",
 * UMDK/CAM pages) step by step, in the pages' order and in the pages' dtypes
 * (fp32 for every dequant / activation / quant step, int32 accumulators),
 * because the block is a quantised pipeline whose result depends on each
 * rounding:
 *   dispatch (§4.1 local token counting, the (bs+1) x E table / prefix-sum
 *            reading of expand_idx, §8.4), stable by flat index t*topk+k;
 *   x quant  (§4.1 "quant fused into dispatch", §7.3 scale stored as
 *            1/dynamicQuantScale; DeepSeek-V4 decode case study, "Freeze the
 *            deployment contract first": W8A8, amax floored, rescaled to 127);
 *   GEMM1    (§3.3 int8 x int8 -> int32);
 *   dequant + SwiGLU (§6.1 EpilogueAtlasA2PerTokenDequantSwiglu:
 *            cast RINT, x weight scale, x per-token scale, left half
 *            x/(1+exp(-x)), right half kept);
 *   requant  (§7.2 BlockQuant: left*right, row amax, scale = amax*(1/127),
 *            q = RINT((h*127)*(1/amax)));
 *   GEMM2    (§3.4) and dequant to bf16 (§6.2 EpilogueAtlasA2PerTokenDequantCombine);
 *   combine  (§4.2 LocalWindowCopy: zero fp32 sum, per k cast, x expert
 *            scale, add, final cast RINT).
 *
 * Readings taken where the pages are silent:
 *   amax floor 1e-4 at both quant points; RNE for every cast; clamp to
 *   [-127, 127]; ids outside [0, E) and masked tokens are skipped; masked
 *   tokens get zero output and zero share_output; the shared expert runs on
 *   every active token with its own smooth scales; smooth scales multiply x
 *   per hidden channel before amax.
 *
 * Signature variants (the pages' input table lists x as bf16 or fp16 and the
 * routed experts' weight scales as fp32, bf16 or fp16; the smooth scales'
 * shape is not given):
 *   fp16 activations: x is read exactly as fp16; y2, output and
 *            share_output take x's dtype (RNE, IEEE overflow to infinity);
 *   16-bit weight scales: widened exactly to fp32, then the same arithmetic;
 *   per-expert smooth scales [E][h]: row (t, k) of expert e is quantised
 *            from x[t] * smooth[e], so x_q and x_scale become per row; the
 *            shared expert keeps its own [h] vector and per-token quant.
 *
 * Compiled with -ffp-contract=off (no fused multiply-add anywhere) so that
 * each fp32 operation rounds once, as the pages' vector instructions do.
 * The transcendental step uses the C library's expf.
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <pthread.h>

#define ORACLE_AMAX_EPS 1e-4f
#define ORACLE_QMAX 127.0f

/* ---------------------------------------------------------------- bf16 -- */
static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* round to nearest, ties to even, on the 16 discarded bits */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- fp16 -- */
/* IEEE binary16 -> binary32, exact: normals by re-biasing the exponent,
 * subnormals as mantissa * 2^-24, infinities and NaNs kept. */
static inline float f16_to_f32(uint16_t b) {
  uint32_t sign = (uint32_t)(b >> 15) << 31;
  int e = (b >> 10) & 0x1F;
  uint32_t m = b & 0x3FFu;
  uint32_t u;
  float f;
  if (e == 0) {
    f = ldexpf((float)m, -24);
    return sign ? -f : f;
  }
  if (e == 31) u = sign | 0x7F800000u | (m << 13);
  else u = sign | ((uint32_t)(e - 15 + 127) << 23) | (m << 13);
  memcpy(&f, &u, 4);
  return f;
}

/* binary32 -> binary16, round to nearest, ties to even.  In the binade
 * [2^e, 2^(e+1)) (e >= -14) fp16 has ulp 2^(e-10): q = rint(|f| / ulp) in
 * [1024, 2048] gives the code ((e + 15) << 10) + q - 1024, where q = 2048
 * carries into the next binade and past e = 15 into infinity.  Below 2^-14
 * the ulp is 2^-24 and q itself is the code (q = 1024 is the least normal). */
static inline uint16_t f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  float a = fabsf(f);
  if (isnan(a)) return (uint16_t)(sign | 0x7E00u);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
  if (a < ldexpf(1.0f, -14)) return (uint16_t)(sign | (uint16_t)rintf(ldexpf(a, 24)));
  int k;
  frexpf(a, &k);            /* a = m * 2^k, m in [0.5, 1): binade e = k - 1 */
  int e = k - 1;
  if (e > 15) return (uint16_t)(sign | 0x7C00u);
  uint32_t q = (uint32_t)rintf(ldexpf(a, 10 - e));
  uint32_t code = ((uint32_t)(e + 15) << 10) + q - 1024u;
  if (code >= 0x7C00u) code = 0x7C00u;
  return (uint16_t)(sign | code);
}

/* activation element (bf16 or fp16 bits) <-> fp32 */
static inline float act_to_f32(uint16_t b, int fp16) { return fp16 ? f16_to_f32(b) : bf16_to_f32(b); }
static inline uint16_t f32_to_act(float f, int fp16) { return fp16 ? f32_to_f16(f) : f32_to_bf16(f); }

/* float -> int8 code: round half to even (rintf under the default mode), clamp */
static inline int8_t f32_to_q(float v) {
  float r = rintf(v);
  if (r > ORACLE_QMAX) r = ORACLE_QMAX;
  if (r < -ORACLE_QMAX) r = -ORACLE_QMAX;
  return (int8_t)r;
}

/* ------------------------------------------------------------ dispatch -- */
/* Counting sort of the active (t, k) pairs by expert, stable by t*topk+k.
 * counts[e], offsets[0..E], row_of[t*topk+k] (-1 when not dispatched),
 * tk_of_row[r] for r < R.  Returns R; *skipped = active pairs whose id is
 * outside [0, E). */
int oracle_dispatch(int bs, int topk, int E, const int32_t* ids, const uint8_t* mask,
                    int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* tk_of_row,
                    int32_t* skipped) {
  int32_t nskip = 0;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int t = 0; t < bs; ++t) {
    int active = mask ? (mask[t] != 0) : 1;
    for (int k = 0; k < topk; ++k) {
      int e = ids[t * topk + k];
      if (!active) continue;
      if (e < 0 || e >= E) { nskip++; continue; }
      counts[e]++;
    }
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int t = 0; t < bs; ++t) {
    int active = mask ? (mask[t] != 0) : 1;
    for (int k = 0; k < topk; ++k) {
      int f = t * topk + k;
      int e = ids[f];
      row_of[f] = -1;
      if (!active || e < 0 || e >= E) continue;
      int r = fill[e]++;
      row_of[f] = r;
      tk_of_row[r] = f;
    }
  }
  free(fill);
  if (skipped) *skipped = nskip;
  return offsets[E];
}

/* --------------------------------------------------------------- quant -- */
/* Per-token dynamic quant of one bf16 row: xs = x * smooth (smooth may be
 * NULL), amax = max(max|xs|, eps), m = 127 / amax, q = rne(xs * m),
 * scale = 1 / m. */
static void quant_row(int h, const uint16_t* x, int fp16, const float* smooth, int8_t* q, float* scale) {
  float* xs = (float*)malloc(sizeof(float) * (size_t)h);
  float amax = 0.0f;
  for (int c = 0; c < h; ++c) {
    float v = act_to_f32(x[c], fp16);
    if (smooth) v = v * smooth[c];
    xs[c] = v;
    float a = fabsf(v);
    if (a > amax) amax = a;
  }
  if (amax < ORACLE_AMAX_EPS) amax = ORACLE_AMAX_EPS;
  float m = ORACLE_QMAX / amax;
  for (int c = 0; c < h; ++c) q[c] = f32_to_q(xs[c] * m);
  *scale = 1.0f / m;
  free(xs);
}
void oracle_quant_row(int h, const uint16_t* x, const float* smooth, int8_t* q, float* scale) {
  quant_row(h, x, 0, smooth, q, scale);
}

/* ---------------------------------------------------------------- GEMM -- */
/* acc[n] = sum_c a[c] * w[n][c] for a row vector a[K] and a row-major
 * weight W[N][K] (output channel n, K contiguous).  |a|,|w| <= 128 and
 * K < 131072 keep every partial sum inside int32. */
int oracle_gemm_row(int N, int K, const int8_t* a, const int8_t* w, int32_t* acc) {
  if (K >= 131072) return -1;
  for (int n = 0; n < N; ++n) {
    const int8_t* wr = w + (size_t)n * (size_t)K;
    int32_t s = 0;
    for (int c = 0; c < K; ++c) s += (int32_t)a[c] * (int32_t)wr[c];
    acc[n] = s;
  }
  return 0;
}

/* ---------------------------------------------------- GEMM1 epilogue -- */
/* y1[n] = (float(acc1[n]) * w1s[n]) * x_scale for n < 2I; gate = y1[0..I),
 * up = y1[I..2I); silu(g) = g / (1 + exp(-g)); h[j] = silu(g[j]) * up[j]. */
void oracle_swiglu_row(int I, const int32_t* acc1, const float* w1s, float x_scale, float* h) {
  for (int j = 0; j < I; ++j) {
    float g = ((float)acc1[j] * w1s[j]) * x_scale;
    float u = ((float)acc1[I + j] * w1s[I + j]) * x_scale;
    float t = expf(-g);
    float d = 1.0f + t;
    float s = g / d;
    h[j] = s * u;
  }
}

/* ------------------------------------------------------------- requant -- */
/* amax = max(max|h|, eps); scale2 = amax * (1/127); q = rne((h*127)*(1/amax)). */
void oracle_requant_row(int I, const float* h, int8_t* q, float* scale2) {
  float amax = 0.0f;
  for (int j = 0; j < I; ++j) {
    float a = fabsf(h[j]);
    if (a > amax) amax = a;
  }
  if (amax < ORACLE_AMAX_EPS) amax = ORACLE_AMAX_EPS;
  float inv127 = 1.0f / ORACLE_QMAX;
  float inv = 1.0f / amax;
  *scale2 = amax * inv127;
  for (int j = 0; j < I; ++j) q[j] = f32_to_q((h[j] * ORACLE_QMAX) * inv);
}

/* ---------------------------------------------------- GEMM2 epilogue -- */
/* y2[j] = rne((float(acc2[j]) * w2s[j]) * scale2) in the activation dtype. */
static void dequant_row(int H, const int32_t* acc2, const float* w2s, float scale2, int fp16, uint16_t* y) {
  for (int j = 0; j < H; ++j) y[j] = f32_to_act(((float)acc2[j] * w2s[j]) * scale2, fp16);
}
void oracle_dequant_bf16_row(int H, const int32_t* acc2, const float* w2s, float scale2, uint16_t* y) {
  dequant_row(H, acc2, w2s, scale2, 0, y);
}

/* ------------------------------------------------------------- combine -- */
/* out[c] = bf16_rne(sum_k float(y2_k[c]) * s_k), sum from 0.0f, k ascending;
 * rows[k] == NULL marks a pair that was not dispatched (it adds nothing). */
static void combine_token(int H, int topk, const uint16_t* const* rows, const float* scales, int fp16,
                          uint16_t* out) {
  for (int c = 0; c < H; ++c) {
    float sum = 0.0f;
    for (int k = 0; k < topk; ++k) {
      if (!rows[k]) continue;
      float p = act_to_f32(rows[k][c], fp16) * scales[k];
      sum = sum + p;
    }
    out[c] = f32_to_act(sum, fp16);
  }
}
void oracle_combine_token(int H, int topk, const uint16_t* const* rows, const float* scales,
                          uint16_t* out) {
  combine_token(H, topk, rows, scales, 0, out);
}

/* Routing weight folded into the GEMM2 row scale (the DeepSeek-V4 decode
 * case study, §2.3: the per-row dequant scale and the routing weight fused
 * into one row scale computed once per row).  Row r of pair (t, k) gets
 * y2'[j] = bf16_rne((float(acc2[j]) * w2s[j]) * (s2 * s_k)), and the combine
 * is the plain sum: out[c] = bf16_rne(sum_k float(y2'_k[c])), from 0.0f, k
 * ascending. */
static void combine_token_folded(int H, int topk, const uint16_t* const* rows, int fp16, uint16_t* out) {
  for (int c = 0; c < H; ++c) {
    float sum = 0.0f;
    for (int k = 0; k < topk; ++k) {
      if (!rows[k]) continue;
      sum = sum + act_to_f32(rows[k][c], fp16);
    }
    out[c] = f32_to_act(sum, fp16);
  }
}
void oracle_combine_token_folded(int H, int topk, const uint16_t* const* rows, uint16_t* out) {
  combine_token_folded(H, topk, rows, 0, out);
}

/* ------------------------------------------------------ whole forward -- */
typedef struct {
  int32_t bs, hidden, num_experts, topk, inter, has_shared;
  const uint16_t* x;                 /* [bs][h] bf16 (or fp16, act_fp16) bits */
  const int32_t* expert_ids;         /* [bs][topk] */
  const float* expert_scales;        /* [bs][topk] */
  const int8_t* const* w1;           /* [E] -> [2I][h]; may be NULL for untouched experts */
  const void* w1_scale;              /* [E][2I], dtype scale_dtype */
  const int8_t* const* w2;           /* [E] -> [h][I] */
  const void* w2_scale;              /* [E][h], dtype scale_dtype */
  const int8_t* share_w1;            /* [2I][h] */
  const float* share_w1_scale;       /* [2I] */
  const int8_t* share_w2;            /* [h][I] */
  const float* share_w2_scale;       /* [h] */
  const float* smooth;               /* [h] ([E][h] with smooth_per_expert) or NULL */
  const float* share_smooth;         /* [h] or NULL */
  const uint8_t* mask;               /* [bs] or NULL */
  const uint8_t* token_sample;       /* [bs] or NULL: compute outputs only where nonzero */
  int32_t threads;
  int32_t fold_routing;              /* 0: default; 1: routing weight folded into the row scale */
  int32_t act_fp16;                  /* 0: x, y2 and outputs bf16; 1: fp16 */
  int32_t scale_dtype;               /* routed weight scales: 0 fp32, 1 bf16, 2 fp16 */
  int32_t smooth_per_expert;         /* 1: smooth is [E][h]; x_q / x_scale are per routed row */
} oracle_args_t;

typedef struct {
  uint16_t* output;          /* [bs][h] */
  uint16_t* share_output;    /* [bs][h] or NULL */
  int32_t* expert_token_nums;/* [E] */
  /* optional intermediates (NULL to skip) */
  int32_t* offsets;          /* [E+1] */
  int32_t* row_of;           /* [bs*topk] */
  int32_t* tk_of_row;        /* [bs*topk] */
  int8_t* x_q;               /* [bs][h] ([R][h] with smooth_per_expert) */
  float* x_scale;            /* [bs] ([R]) */
  int8_t* xs_q;              /* [bs][h] shared-expert quant */
  float* xs_scale;           /* [bs] */
  int32_t* acc1;             /* [R][2I] routed rows */
  float* h_act;              /* [R][I] */
  int8_t* x2;                /* [R][I] */
  float* s2;                 /* [R] */
  int32_t* acc2;             /* [R][h] */
  uint16_t* y2;              /* [R][h] */
  int32_t* share_acc1;       /* [bs][2I] (rows of inactive tokens untouched) */
  float* share_h;            /* [bs][I] */
  int8_t* share_x2;          /* [bs][I] */
  float* share_s2;           /* [bs] */
  int32_t* share_acc2;       /* [bs][h] */
  int32_t skipped;           /* out: active pairs with an id outside [0, E) */
  int32_t R;                 /* out: dispatched rows */
} oracle_out_t;

typedef struct {
  const oracle_args_t* a;
  oracle_out_t* o;
  int job;          /* 0 quant, 1 routed rows, 2 shared rows, 3 combine */
  int begin, end;
  const int32_t* tk_of_row;
  const int32_t* row_of;
  const int8_t* xq;  const float* xsc;
  const int8_t* sq;  const float* ssc;
  const float* w1s; const float* w2s;   /* routed weight scales widened to fp32 */
  uint16_t* y2;
  int rc;
} work_t;

static void widen_scales(const void* src, int dtype, size_t n, float* dst) {
  for (size_t i = 0; i < n; ++i) {
    if (dtype == 0) dst[i] = ((const float*)src)[i];
    else if (dtype == 1) dst[i] = bf16_to_f32(((const uint16_t*)src)[i]);
    else dst[i] = f16_to_f32(((const uint16_t*)src)[i]);
  }
}

/* one routed or shared row: GEMM1 -> SwiGLU -> requant -> GEMM2 -> dequant;
 * route_scale (non-NULL only for routed rows in the folded mode) multiplies
 * the requant scale once before the GEMM2 dequant */
static int expert_row(int h, int I, int fp16, const int8_t* xrow, float xscale,
                      const int8_t* w1, const float* w1s, const int8_t* w2, const float* w2s,
                      const float* route_scale,
                      int32_t* acc1_out, float* h_out, int8_t* x2_out, float* s2_out,
                      int32_t* acc2_out, uint16_t* y_out) {
  int32_t* acc1 = (int32_t*)malloc(sizeof(int32_t) * (size_t)(2 * I));
  float* hv = (float*)malloc(sizeof(float) * (size_t)I);
  int8_t* q2 = (int8_t*)malloc((size_t)I);
  int32_t* acc2 = (int32_t*)malloc(sizeof(int32_t) * (size_t)h);
  float s2;
  int rc = oracle_gemm_row(2 * I, h, xrow, w1, acc1);
  if (rc == 0) {
    oracle_swiglu_row(I, acc1, w1s, xscale, hv);
    oracle_requant_row(I, hv, q2, &s2);
    rc = oracle_gemm_row(h, I, q2, w2, acc2);
  }
  if (rc == 0) {
    dequant_row(h, acc2, w2s, route_scale ? s2 * (*route_scale) : s2, fp16, y_out);
    if (acc1_out) memcpy(acc1_out, acc1, sizeof(int32_t) * (size_t)(2 * I));
    if (h_out) memcpy(h_out, hv, sizeof(float) * (size_t)I);
    if (x2_out) memcpy(x2_out, q2, (size_t)I);
    if (s2_out) *s2_out = s2;
    if (acc2_out) memcpy(acc2_out, acc2, sizeof(int32_t) * (size_t)h);
  }
  free(acc1); free(hv); free(q2); free(acc2);
  return rc;
}

static void* worker(void* p) {
  work_t* w = (work_t*)p;
  const oracle_args_t* a = w->a;
  oracle_out_t* o = w->o;
  int h = a->hidden, I = a->inter, K = a->topk;
  w->rc = 0;
  for (int i = w->begin; i < w->end && w->rc == 0; ++i) {
    if (w->job == 0) {               /* quant token i (routed: only with one [h] smooth vector) */
      const uint16_t* xt = a->x + (size_t)i * h;
      if (!a->smooth_per_expert)
        quant_row(h, xt, a->act_fp16, a->smooth, (int8_t*)w->xq + (size_t)i * h, (float*)w->xsc + i);
      if (a->has_shared)
        quant_row(h, xt, a->act_fp16, a->share_smooth, (int8_t*)w->sq + (size_t)i * h, (float*)w->ssc + i);
    } else if (w->job == 1) {        /* routed row i */
      int f = w->tk_of_row[i];
      int t = f / K;
      if (a->token_sample && !a->token_sample[t]) continue;
      int e = a->expert_ids[f];
      if (!a->w1[e] || !a->w2[e]) { w->rc = -2; break; }
      /* the row's int8 operand: token t's codes, or (per-expert smooth) row
       * i's own quant of x[t] * smooth[e] */
      const int8_t* xrow = w->xq + (size_t)t * h;
      float xs = w->xsc[t];
      if (a->smooth_per_expert) {
        int8_t* q = (int8_t*)w->xq + (size_t)i * h;
        quant_row(h, a->x + (size_t)t * h, a->act_fp16, a->smooth + (size_t)e * h, q, (float*)w->xsc + i);
        xrow = q;
        xs = w->xsc[i];
      }
      w->rc = expert_row(h, I, a->act_fp16, xrow, xs,
                         a->w1[e], w->w1s + (size_t)e * 2 * I, a->w2[e], w->w2s + (size_t)e * h,
                         a->fold_routing ? a->expert_scales + f : NULL,
                         o->acc1 ? o->acc1 + (size_t)i * 2 * I : NULL,
                         o->h_act ? o->h_act + (size_t)i * I : NULL,
                         o->x2 ? o->x2 + (size_t)i * I : NULL,
                         o->s2 ? o->s2 + i : NULL,
                         o->acc2 ? o->acc2 + (size_t)i * h : NULL,
                         w->y2 + (size_t)i * h);
    } else if (w->job == 2) {        /* shared expert on token i */
      int active = a->mask ? (a->mask[i] != 0) : 1;
      uint16_t* so = o->share_output + (size_t)i * h;
      if (a->token_sample && !a->token_sample[i]) continue;
      if (!active) { memset(so, 0, sizeof(uint16_t) * (size_t)h); continue; }
      w->rc = expert_row(h, I, a->act_fp16, w->sq + (size_t)i * h, w->ssc[i],
                         a->share_w1, a->share_w1_scale, a->share_w2, a->share_w2_scale, NULL,
                         o->share_acc1 ? o->share_acc1 + (size_t)i * 2 * I : NULL,
                         o->share_h ? o->share_h + (size_t)i * I : NULL,
                         o->share_x2 ? o->share_x2 + (size_t)i * I : NULL,
                         o->share_s2 ? o->share_s2 + i : NULL,
                         o->share_acc2 ? o->share_acc2 + (size_t)i * h : NULL,
                         so);
    } else {                          /* combine token i */
      int active = a->mask ? (a->mask[i] != 0) : 1;
      uint16_t* out = o->output + (size_t)i * h;
      if (a->token_sample && !a->token_sample[i]) continue;
      if (!active) { memset(out, 0, sizeof(uint16_t) * (size_t)h); continue; }
      const uint16_t* rows[64];
      for (int k = 0; k < K; ++k) {
        int r = w->row_of[i * K + k];
        rows[k] = r >= 0 ? w->y2 + (size_t)r * h : NULL;
      }
      if (a->fold_routing) combine_token_folded(h, K, rows, a->act_fp16, out);
      else combine_token(h, K, rows, a->expert_scales + (size_t)i * K, a->act_fp16, out);
    }
  }
  return NULL;
}

static int run_parallel(const oracle_args_t* a, oracle_out_t* o, int job, int n, work_t* tmpl) {
  int T = a->threads > 0 ? a->threads : 1;
  if (T > 256) T = 256;
  if (T > n) T = n > 0 ? n : 1;
  pthread_t tid[256];
  work_t w[256];
  int started[256];
  int per = n / T, extra = n % T, b = 0;
  for (int i = 0; i < T; ++i) {
    w[i] = *tmpl;
    w[i].a = a; w[i].o = o; w[i].job = job;
    w[i].begin = b; b += per + (i < extra ? 1 : 0); w[i].end = b;
    started[i] = pthread_create(&tid[i], NULL, worker, &w[i]) == 0;
    if (!started[i]) worker(&w[i]);
  }
  int rc = 0;
  for (int i = 0; i < T; ++i) {
    if (started[i]) pthread_join(tid[i], NULL);
    if (w[i].rc) rc = w[i].rc;
  }
  return rc;
}

/* Whole block.  Returns 0, -1 (K too large for int32), -2 (missing weights of
 * a touched expert), -3 (bad arguments). */
int oracle_forward(const oracle_args_t* a, oracle_out_t* o) {
  int bs = a->bs, h = a->hidden, E = a->num_experts, K = a->topk, I = a->inter;
  if (bs < 0 || h <= 0 || E <= 0 || K <= 0 || K > 64 || I <= 0) return -3;
  if (a->has_shared && (!a->share_w1 || !a->share_w2 || !o->share_output)) return -3;
  size_t nf = (size_t)bs * K;
  int32_t* offsets = o->offsets ? o->offsets : (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t* row_of = o->row_of ? o->row_of : (int32_t*)malloc(sizeof(int32_t) * (nf ? nf : 1));
  int32_t* tk_of_row = o->tk_of_row ? o->tk_of_row : (int32_t*)malloc(sizeof(int32_t) * (nf ? nf : 1));
  int R = oracle_dispatch(bs, K, E, a->expert_ids, a->mask, o->expert_token_nums, offsets,
                          row_of, tk_of_row, &o->skipped);
  o->R = R;

  if (a->scale_dtype < 0 || a->scale_dtype > 2) return -3;
  size_t nq = a->smooth_per_expert ? (size_t)R : (size_t)bs;   /* quantised routed rows */
  int8_t* xq = o->x_q ? o->x_q : (int8_t*)malloc(nq * h + 1);
  float* xsc = o->x_scale ? o->x_scale : (float*)malloc(sizeof(float) * (nq + 1));
  /* routed weight scales in fp32 (a 16-bit scale widens exactly) */
  float* w1s = (float*)malloc(sizeof(float) * (size_t)E * 2 * I);
  float* w2s = (float*)malloc(sizeof(float) * (size_t)E * h);
  widen_scales(a->w1_scale, a->scale_dtype, (size_t)E * 2 * I, w1s);
  widen_scales(a->w2_scale, a->scale_dtype, (size_t)E * h, w2s);
  int8_t* sq = NULL; float* ssc = NULL;
  if (a->has_shared) {
    sq = o->xs_q ? o->xs_q : (int8_t*)malloc((size_t)bs * h + 1);
    ssc = o->xs_scale ? o->xs_scale : (float*)malloc(sizeof(float) * (size_t)(bs + 1));
  }
  uint16_t* y2 = o->y2 ? o->y2 : (uint16_t*)malloc(sizeof(uint16_t) * ((size_t)R * h + 1));

  work_t tmpl;
  memset(&tmpl, 0, sizeof(tmpl));
  tmpl.tk_of_row = tk_of_row; tmpl.row_of = row_of;
  tmpl.xq = xq; tmpl.xsc = xsc; tmpl.sq = sq; tmpl.ssc = ssc; tmpl.y2 = y2;
  tmpl.w1s = w1s; tmpl.w2s = w2s;

  int rc = 0;
  if (bs > 0) rc = run_parallel(a, o, 0, bs, &tmpl);               /* quant every token */
  if (rc == 0 && R > 0) rc = run_parallel(a, o, 1, R, &tmpl);      /* routed rows */
  if (rc == 0 && a->has_shared && bs > 0) rc = run_parallel(a, o, 2, bs, &tmpl);
  if (rc == 0 && bs > 0) rc = run_parallel(a, o, 3, bs, &tmpl);    /* combine */

  if (!o->offsets) free(offsets);
  if (!o->row_of) free(row_of);
  if (!o->tk_of_row) free(tk_of_row);
  if (!o->x_q) free(xq);
  if (!o->x_scale) free(xsc);
  if (a->has_shared && !o->xs_q) free(sq);
  if (a->has_shared && !o->xs_scale) free(ssc);
  if (!o->y2) free(y2);
  free(w1s); free(w2s);
  return rc;
}

/* exported helpers for pins */
float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }
float oracle_f16_to_f32(uint16_t b) { return f16_to_f32(b); }
uint16_t oracle_f32_to_f16(float f) { return f32_to_f16(f); }
uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16(f); }
int oracle_sizeof_args(void) { return (int)sizeof(oracle_args_t); }
int oracle_sizeof_out(void) { return (int)sizeof(oracle_out_t); }
