/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for MoE token
 * dispatch and combine.  TEST INFRASTRUCTURE ONLY (see moe_oracle.h).
 *
 * Every function is the plain definition written out as loops.  There is no
 * blocking, fusion or reordering.  Build with -O2 -ffp-contract=off and
 * without -ffast-math, so that float arithmetic is IEEE binary32 with
 * round-to-nearest-even and only the fmaf() calls below fuse.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats, written from the format definitions.                      */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: the value is exact. */
float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Keep the upper 16 bits; round the dropped lower 16 bits to nearest, ties
 * to the even upper half.  A carry out of the mantissa moves to the next
 * binade (and to infinity past the largest finite value), as IEEE does. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if (isnan(f)) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* OCP 8-bit floating point, E4M3 ("FN"): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent field 0 holds subnormals m * 2^-9;
 * field 15 with mantissa 7 is NaN; there is no infinity; the largest finite
 * magnitude is 1.75 * 2^8 = 448. */
float oracle_e4m3_to_f32(uint8_t q) {
  int sign = (q & 0x80) ? -1 : 1;
  int ex = (q >> 3) & 0xF;
  int m = q & 0x7;
  if (ex == 0xF && m == 0x7) return NAN;
  double v;
  if (ex == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + (double)m / 8.0, ex - 7);
  return (float)(sign * v);
}

/* Round |f| to the E4M3 grid: find the spacing of the grid in the binade of
 * |f| (2^-9 in the subnormal range, 2^(k-3) in [2^k, 2^(k+1)) for k >= -6),
 * round |f| / spacing to an integer with ties to even (rint() in the
 * default rounding mode), and encode the result.  Magnitudes >= 448 saturate
 * to 448: those in [448, 464) round to 448 and those above would overflow. */
uint8_t oracle_f32_to_e4m3(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint8_t sign = (u >> 31) ? 0x80 : 0x00;
  if (isnan(f)) return (uint8_t)(0x7F | sign);
  double a = fabs((double)f);
  if (a >= 448.0) return (uint8_t)(0x7E | sign);
  if (a == 0.0) return sign;

  int e2;
  (void)frexp(a, &e2);       /* a = m * 2^e2, m in [0.5, 1) */
  int k = e2 - 1;            /* a in [2^k, 2^(k+1)) */
  if (k < -6) k = -6;        /* subnormals share the spacing of 2^-6's binade */
  double spacing = ldexp(1.0, k - 3);
  double n = rint(a / spacing); /* exact quotient; ties to even */
  double v = n * spacing;       /* the rounded magnitude, exactly */

  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) {     /* subnormal: v = m * 2^-9, m in 1..7 */
    int m = (int)(v / ldexp(1.0, -9));
    return (uint8_t)(sign | m);
  }
  (void)frexp(v, &e2);
  int kv = e2 - 1;                                 /* v in [2^kv, 2^(kv+1)) */
  int m = (int)((v / ldexp(1.0, kv) - 1.0) * 8.0); /* 0..7, exact */
  return (uint8_t)(sign | ((kv + 7) << 3) | m);
}

void oracle_bf16_to_f32_n(int64_t n, const uint16_t *in, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(in[i]);
}
void oracle_f32_to_bf16_n(int64_t n, const float *in, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}
void oracle_e4m3_to_f32_n(int64_t n, const uint8_t *in, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f32(in[i]);
}
void oracle_f32_to_e4m3_n(int64_t n, const float *in, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Plan.                                                                     */
/* ------------------------------------------------------------------------ */

/* "Efficient and portable mixture-of-experts communication", Dispatch: the
 * sender counts how many tokens each expert receives, and the receiver keeps
 * (source rank, expert, token) so that combine knows where each row goes.
 * "Enabling trillion-parameter models on AWS EFA", Send and Receive Buffers /
 * Dispatch and Combine: per-expert counts are exchanged first and a
 * cumulative sum of them gives each sender's offset inside the receiver's
 * contiguous buffer.
 *
 * Reading taken for the slot order (the pages' receiver order is not
 * deterministic): stable by (source logical rank, token, k).  Ranks are
 * contiguous token ranges, so this is ascending global (g, k) order.
 *
 *   expert_num_tokens[e]      = #{(g,k) : idx[g,k] = e}
 *   expert_rank_offsets[e][r] = #{(g,k) : idx[g,k] = e and g < r*T}, r = 0..R
 *   slot_of[g,k]              = #{(g',k') before (g,k) : idx[g',k'] = idx[g,k]}
 *   src_of[e][slot_of[g,k]]   = g*K + k
 */
int oracle_plan(int R, int T, int E, int K, int cap, const int32_t *topk_idx,
                int32_t *expert_num_tokens, int32_t *expert_rank_offsets,
                int32_t *slot_of, int32_t *src_of) {
  if (R <= 0 || T < 0 || E <= 0 || K <= 0 || cap <= 0) return ORACLE_BAD_SHAPE;
  const int64_t N = (int64_t)R * T;

  for (int64_t i = 0; i < N * K; ++i)
    if (topk_idx[i] < 0 || topk_idx[i] >= E) return ORACLE_BAD_EXPERT;

  /* counts */
  for (int e = 0; e < E; ++e) expert_num_tokens[e] = 0;
  for (int64_t g = 0; g < N; ++g)
    for (int k = 0; k < K; ++k) expert_num_tokens[topk_idx[g * K + k]] += 1;

  /* per-rank offsets, straight from the definition */
  for (int e = 0; e < E; ++e)
    for (int r = 0; r <= R; ++r) expert_rank_offsets[(int64_t)e * (R + 1) + r] = 0;
  for (int r = 0; r <= R; ++r)
    for (int64_t g = 0; g < (int64_t)r * T; ++g)
      for (int k = 0; k < K; ++k)
        expert_rank_offsets[(int64_t)topk_idx[g * K + k] * (R + 1) + r] += 1;

  /* stable slots and return addresses */
  int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  if (!fill) abort();
  int status = ORACLE_OK;
  for (int64_t g = 0; g < N; ++g) {
    for (int k = 0; k < K; ++k) {
      int e = topk_idx[g * K + k];
      int s = fill[e];
      fill[e] += 1;
      slot_of[g * K + k] = s;
      if (s < cap) src_of[(int64_t)e * cap + s] = (int32_t)(g * K + k);
      else status = ORACLE_CAPACITY;
    }
  }
  free(fill);
  return status;
}

/* "Lower latency and higher throughput with multi-node DeepSeek deployment",
 * CUDA Graph: data-parallel groups run different batch sizes, and the
 * all-to-all kernels let them do so without padding every group to the
 * largest batch.  "Efficient and portable mixture-of-experts communication",
 * Portable Kernels: the number of tokens a group sends is bounded by a fixed
 * maximum per group (here T).
 *
 * Readings taken: rank r holds num_tokens[r] valid tokens (clamped to
 * [0, T]); an expert id of -1 marks an entry that is not routed.  Only
 * routed entries are counted and get slots, in the same stable (rank, token,
 * k) order; the others get slot_of = -1. */
static int routed_entry(int T, int K, const int32_t *num_tokens, const int32_t *topk_idx,
                        int64_t g, int k) {
  int64_t r = g / T, t = g % T;
  if (num_tokens) {
    int64_t nt = num_tokens[r];
    if (nt < 0) nt = 0;
    if (nt > T) nt = T;
    if (t >= nt) return 0;
  }
  return topk_idx[g * K + k] != -1;
}

int oracle_plan_masked(int R, int T, int E, int K, int cap, const int32_t *topk_idx,
                       const int32_t *num_tokens, int32_t *expert_num_tokens,
                       int32_t *expert_rank_offsets, int32_t *slot_of, int32_t *src_of) {
  if (R <= 0 || T < 0 || E <= 0 || K <= 0 || cap <= 0) return ORACLE_BAD_SHAPE;
  const int64_t N = (int64_t)R * T;

  for (int64_t g = 0; g < N; ++g)
    for (int k = 0; k < K; ++k)
      if (routed_entry(T, K, num_tokens, topk_idx, g, k) &&
          (topk_idx[g * K + k] < 0 || topk_idx[g * K + k] >= E))
        return ORACLE_BAD_EXPERT;

  for (int e = 0; e < E; ++e) expert_num_tokens[e] = 0;
  for (int64_t g = 0; g < N; ++g)
    for (int k = 0; k < K; ++k)
      if (routed_entry(T, K, num_tokens, topk_idx, g, k))
        expert_num_tokens[topk_idx[g * K + k]] += 1;

  for (int e = 0; e < E; ++e)
    for (int r = 0; r <= R; ++r) expert_rank_offsets[(int64_t)e * (R + 1) + r] = 0;
  for (int r = 0; r <= R; ++r)
    for (int64_t g = 0; g < (int64_t)r * T; ++g)
      for (int k = 0; k < K; ++k)
        if (routed_entry(T, K, num_tokens, topk_idx, g, k))
          expert_rank_offsets[(int64_t)topk_idx[g * K + k] * (R + 1) + r] += 1;

  int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  if (!fill) abort();
  int status = ORACLE_OK;
  for (int64_t g = 0; g < N; ++g) {
    for (int k = 0; k < K; ++k) {
      if (!routed_entry(T, K, num_tokens, topk_idx, g, k)) {
        slot_of[g * K + k] = -1;
        continue;
      }
      int e = topk_idx[g * K + k];
      int s = fill[e];
      fill[e] += 1;
      slot_of[g * K + k] = s;
      if (s < cap) src_of[(int64_t)e * cap + s] = (int32_t)(g * K + k);
      else status = ORACLE_CAPACITY;
    }
  }
  free(fill);
  return status;
}

/* ------------------------------------------------------------------------ */
/* Dispatch.                                                                 */
/* ------------------------------------------------------------------------ */

/* Each token row is written to every (expert, slot) it is routed to. */
void oracle_dispatch_bf16(int N, int H, int E, int K, int cap,
                          const uint16_t *x, const int32_t *topk_idx,
                          const int32_t *slot_of, uint16_t *expert_x) {
  for (int64_t g = 0; g < N; ++g) {
    for (int k = 0; k < K; ++k) {
      int e = topk_idx[g * K + k];
      int s = slot_of[g * K + k];
      if (e < 0 || e >= E || s < 0 || s >= cap) continue;
      uint16_t *dst = expert_x + ((int64_t)e * cap + s) * H;
      for (int h = 0; h < H; ++h) dst[h] = x[g * H + h];
    }
  }
}

/* "Lower latency and higher throughput with multi-node DeepSeek
 * deployment", Quantization: activations are quantised on the fly with one
 * scale per 128-element vector along the hidden dimension (scale shape
 * M x ceil_div(K, 128) for an M x K activation), found from the largest
 * absolute value of the block.
 *
 * Readings taken (the pages fix only "absmax per 128 elements" and fp8):
 *   blocks  = ceil_div(H, 128); the last block holds the H % 128 elements
 *             left over when H is not a multiple of 128 (the scale shape
 *             M x ceil_div(K, 128) above)
 *   amax  = max |x_i| over the block (exact in fp32)
 *   scale = amax / 448   (IEEE binary32 division; 448 = largest E4M3)
 *   q_i   = e4m3(x_i / scale)   (binary32 division, then RNE + saturate)
 *   a block of zeros has scale 0 and q_i = +0.
 */
void oracle_quant_row_e4m3(int H, const uint16_t *row, uint8_t *q,
                           float *scale) {
  const int nb = (H + 127) / 128;   /* ceil_div(H, 128): the last block may be short */
  for (int b = 0; b < nb; ++b) {
    const int end = (b + 1) * 128 < H ? (b + 1) * 128 : H;
    float amax = 0.0f;
    for (int i = b * 128; i < end; ++i) {
      float a = fabsf(oracle_bf16_to_f32(row[i]));
      if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    scale[b] = s;
    for (int i = b * 128; i < end; ++i) {
      if (amax == 0.0f) q[i] = 0x00;
      else q[i] = oracle_f32_to_e4m3(oracle_bf16_to_f32(row[i]) / s);
    }
  }
}

void oracle_dispatch_fp8(int N, int H, int E, int K, int cap,
                         const uint16_t *x, const int32_t *topk_idx,
                         const int32_t *slot_of, uint8_t *expert_x,
                         float *expert_x_scale) {
  const int nb = (H + 127) / 128;
  uint8_t *q = (uint8_t *)malloc((size_t)H);
  float *sc = (float *)malloc((size_t)nb * sizeof(float));
  if (!q || !sc) abort();
  for (int64_t g = 0; g < N; ++g) {
    oracle_quant_row_e4m3(H, x + g * H, q, sc);
    for (int k = 0; k < K; ++k) {
      int e = topk_idx[g * K + k];
      int s = slot_of[g * K + k];
      if (e < 0 || e >= E || s < 0 || s >= cap) continue;
      int64_t row = (int64_t)e * cap + s;
      for (int h = 0; h < H; ++h) expert_x[row * H + h] = q[h];
      for (int b = 0; b < nb; ++b) expert_x_scale[row * nb + b] = sc[b];
    }
  }
  free(q);
  free(sc);
}

/* ------------------------------------------------------------------------ */
/* Combine.                                                                  */
/* ------------------------------------------------------------------------ */

/* "Efficient and portable mixture-of-experts communication", Introduction and
 * Combine: the output of a token is the sum of its experts' outputs, each
 * multiplied by the router weight, computed where the token came from, from
 * 16-bit expert outputs.
 *
 * Reading taken for the arithmetic (not fixed by the pages): one fp32
 * accumulator per element starting at +0, one fused multiply-add per k in
 * ascending k, and a single round to bf16 at the end. */
void oracle_combine(int N, int H, int E, int K, int cap,
                    const uint16_t *expert_y, const int32_t *topk_idx,
                    const int32_t *slot_of, const float *topk_weights,
                    uint16_t *y) {
  for (int64_t g = 0; g < N; ++g) {
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int k = 0; k < K; ++k) {
        int e = topk_idx[g * K + k];
        int s = slot_of[g * K + k];
        if (e < 0 || e >= E || s < 0 || s >= cap) continue;
        float v = oracle_bf16_to_f32(expert_y[((int64_t)e * cap + s) * H + h]);
        acc = fmaf(topk_weights[g * K + k], v, acc);
      }
      y[g * H + h] = oracle_f32_to_bf16(acc);
    }
  }
}

/* "Lower latency and higher throughput with multi-node DeepSeek
 * deployment", Expert Parallelism and Compute/Communication Overlap: each
 * token also goes through a shared expert, whose output is added to the
 * routed experts' weighted sum (and can be computed while dispatch is in
 * flight).  Reading taken: the shared output (bf16) seeds the fp32
 * accumulator, the routed terms follow in ascending k, one final rounding. */
void oracle_combine_shared(int N, int H, int E, int K, int cap,
                           const uint16_t *expert_y, const int32_t *topk_idx,
                           const int32_t *slot_of, const float *topk_weights,
                           const uint16_t *shared, uint16_t *y) {
  for (int64_t g = 0; g < N; ++g) {
    for (int h = 0; h < H; ++h) {
      float acc = oracle_bf16_to_f32(shared[g * H + h]);
      for (int k = 0; k < K; ++k) {
        int e = topk_idx[g * K + k];
        int s = slot_of[g * K + k];
        if (e < 0 || e >= E || s < 0 || s >= cap) continue;
        float v = oracle_bf16_to_f32(expert_y[((int64_t)e * cap + s) * H + h]);
        acc = fmaf(topk_weights[g * K + k], v, acc);
      }
      y[g * H + h] = oracle_f32_to_bf16(acc); /* shared + routed, one rounding */
    }
  }
}

/* "Efficient and portable mixture-of-experts communication", Introduction:
 * the router is a small linear layer producing a probability distribution
 * over experts; the experts with the K highest scores are chosen and the
 * output is their average weighted by the router's probabilities.  "Lower
 * latency and higher throughput with multi-node DeepSeek deployment", MoE
 * Router: a sort that tracks the indices of the sorted elements; the sparse
 * kernels consume the top-K indices and scores directly.
 *
 * Readings taken: order by logit, descending, ties by lower expert index;
 * weights = softmax over the K chosen logits (the renormalised top-K of the
 * full softmax), exp(l_k - l_max) / sum, in fp64, rounded once to fp32. */
static const float *router_row;

static int router_cmp(const void *a, const void *b) {
  const int ia = *(const int *)a, ib = *(const int *)b;
  const float la = router_row[ia], lb = router_row[ib];
  if (la > lb) return -1;
  if (la < lb) return 1;
  return (ia > ib) - (ia < ib);
}

void oracle_router_topk(int N, int E, int K, const float *logits, int32_t *topk_idx,
                        float *topk_weights) {
  int *order = (int *)malloc((size_t)E * sizeof(int));
  double *z = (double *)malloc((size_t)K * sizeof(double));
  if (!order || !z) abort();
  for (int64_t g = 0; g < N; ++g) {
    router_row = logits + g * E;
    for (int e = 0; e < E; ++e) order[e] = e;
    qsort(order, (size_t)E, sizeof(int), router_cmp);
    const double m = (double)router_row[order[0]];
    double sum = 0.0;
    for (int k = 0; k < K; ++k) {
      z[k] = exp((double)router_row[order[k]] - m);
      sum += z[k];
    }
    for (int k = 0; k < K; ++k) {
      topk_idx[g * K + k] = order[k];
      topk_weights[g * K + k] = (float)(z[k] / sum);
    }
  }
  free(order);
  free(z);
}

/* ------------------------------------------------------------------------ */
/* Activation and re-quantisation between the expert GEMMs.                  */
/* ------------------------------------------------------------------------ */

/* e^x in binary32.  The pages fix no algorithm; for the quantised bytes to be
 * reproducible bit for bit, this library fixes one, the classic Cody-Waite
 * scheme (Cody & Waite, "Software Manual for the Elementary Functions"):
 *   n = rint(x * log2(e)),  r = x - n*ln2_hi - n*ln2_lo   (ln2_hi has 16
 *   significant bits, so n*ln2_hi is exact for |n| < 256),
 *   e^r ~ sum_{k<=7} r^k / k!  (Horner with fmaf; truncation < 1e-8 on
 *   |r| <= ln2/2),  e^x = e^r * 2^n  (2^n built exactly).
 * Every step is one IEEE binary32 operation, so any implementation that
 * executes the same steps gets the same bits. */
float oracle_exp_f32(float x) {
  if (x > 88.72f) return INFINITY;
  if (x < -87.33f) return 0.0f;
  const float ln2_hi = 0.693145751953125f;      /* 0x3F317200 */
  const float ln2_lo = 1.42860677e-06f;         /* 0x35BFBE8E */
  const float log2e = 1.44269502f;              /* 0x3FB8AA3B */
  const float n = rintf(x * log2e);
  float r = fmaf(-n, ln2_hi, x);
  r = fmaf(-n, ln2_lo, r);
  float p = 1.98412701e-04f;                     /* 1/7!  0x39500D01 */
  p = fmaf(p, r, 1.38888892e-03f);               /* 1/6!  0x3AB60B61 */
  p = fmaf(p, r, 8.33333377e-03f);               /* 1/5!  0x3C088889 */
  p = fmaf(p, r, 4.16666679e-02f);               /* 1/4!  0x3D2AAAAB */
  p = fmaf(p, r, 1.66666672e-01f);               /* 1/3!  0x3E2AAAAB */
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n;
  if (ni > 127) {                                /* 2^128 is not a float */
    p = p * 2.0f;
    ni -= 1;
  }
  uint32_t bits = (uint32_t)(ni + 127) << 23;
  float two_n;
  memcpy(&two_n, &bits, sizeof two_n);
  return p * two_n;
}

float oracle_silu_f32(float g) {
  return g / (1.0f + oracle_exp_f32(-g));
}

/* "Lower latency and higher throughput with multi-node DeepSeek
 * deployment", Quantization: the SiLU kernel works on activations split
 * along the hidden dimension, quantises them with one scale per 128
 * elements from the absolute maximum, and, to stay valid inside CUDA
 * graphs, reads the per-expert token counts to decide which rows hold
 * tokens instead of relying on the buffer sizes.  Reading taken: the first
 * half of each expert_h row is the gate projection, the second the up
 * projection; a = SiLU(gate) * up in binary32; quantisation as in
 * oracle_quant_row_e4m3, applied to a. */
void oracle_silu_mul_quant(int E, int cap, int I, const uint16_t *expert_h,
                           const int32_t *expert_num_tokens, uint8_t *act_q,
                           float *act_scale) {
  float *a = (float *)malloc((size_t)I * sizeof(float));
  if (!a) abort();
  const int nb = (I + 127) / 128;   /* ceil_div(I, 128): the last block may be short */
  for (int e = 0; e < E; ++e) {
    int rows = expert_num_tokens[e];
    if (rows < 0) rows = 0;
    if (rows > cap) rows = cap;
    for (int s = 0; s < rows; ++s) {
      const int64_t row = (int64_t)e * cap + s;
      const uint16_t *h = expert_h + row * 2 * I;
      for (int i = 0; i < I; ++i) {
        const float g = oracle_bf16_to_f32(h[i]);
        const float u = oracle_bf16_to_f32(h[I + i]);
        a[i] = oracle_silu_f32(g) * u;
      }
      for (int b = 0; b < nb; ++b) {
        const int end = (b + 1) * 128 < I ? (b + 1) * 128 : I;
        float amax = 0.0f;
        for (int i = b * 128; i < end; ++i) {
          const float v = fabsf(a[i]);
          if (v > amax) amax = v;
        }
        const float sc = amax / 448.0f;
        act_scale[row * nb + b] = sc;
        for (int i = b * 128; i < end; ++i)
          act_q[row * I + i] = (amax == 0.0f) ? 0x00 : oracle_f32_to_e4m3(a[i] / sc);
      }
    }
  }
  free(a);
}
