/*
 * moe_oracle.h -- plain, slow, single-threaded CPU oracle for MoE token
 * dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The product
 * path (the CUDA library under combine_moe_dispatch_gb300/) never calls it,
 * shares no code with it, and fails loudly when its own extension is missing.
 *
 * What is computed, and where the pages define it:
 *  - Routing: each token goes to K experts and the layer output is the
 *    router-weighted sum of the expert outputs ("Efficient and portable
 *    mixture-of-experts communication", Introduction).
 *  - Plan: per-expert token counts (in the pages a single warp per block
 *    tallies them while the others pack; same page, Dispatch), the cumulative
 *    sum of those counts giving packing offsets ("Enabling trillion-parameter
 *    models on AWS EFA", Dispatch and Combine; Send and Receive Buffers), and
 *    return addresses (source rank, expert, token index) kept for combine
 *    ("Efficient and portable mixture-of-experts communication", Dispatch).
 *  - Dispatch payload: a bf16 copy, or fp8 with one scale per 128-element
 *    activation vector computed on the fly from the absolute maximum ("Lower
 *    latency and higher throughput with multi-node DeepSeek deployment",
 *    Quantization).
 *  - Combine: 16-bit un-quantised expert outputs, weighted average computed
 *    at the receiver ("Efficient and portable mixture-of-experts
 *    communication", Combine).
 *
 * Readings where the pages leave a step open (slot order, scale formula,
 * rounding, accumulation order) are stated next to each function.
 *
 * Layouts (all row-major, global token id g = r*T + t, N = R*T):
 *   topk_idx      [N, K]        int32
 *   topk_weights  [N, K]        float
 *   x             [N, H]        bf16 bit patterns (uint16)
 *   expert_num_tokens [E]       int32
 *   expert_rank_offsets [E, R+1] int32
 *   slot_of       [N, K]        int32
 *   src_of        [E, cap]      int32 (only [0, count) written)
 *   expert_x      [E, cap, H]   bf16 bits, or e4m3 bytes
 *   expert_x_scale [E, cap, H/128] float
 *   expert_y      [E, cap, H]   bf16 bits
 *   y             [N, H]        bf16 bits
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Result codes of the oracle (its own numbering; not shared with the CUDA
 * library). */
enum {
  ORACLE_OK = 0,
  ORACLE_BAD_EXPERT = 1, /* some topk_idx outside [0, E) */
  ORACLE_CAPACITY = 2,   /* some expert receives more than cap rows */
  ORACLE_BAD_SHAPE = 3   /* non-positive or inconsistent sizes */
};

/* ---- number formats ---------------------------------------------------- */
/* bf16 bits -> float (exact). */
float oracle_bf16_to_f32(uint16_t b);
/* float -> bf16 bits, round to nearest, ties to even; NaN -> 0x7FC0 with the
 * input's sign. */
uint16_t oracle_f32_to_bf16(float f);
/* OCP FP8 E4M3 ("FN") byte -> float (exact; 0x7F/0xFF -> NaN). */
float oracle_e4m3_to_f32(uint8_t q);
/* float -> OCP FP8 E4M3 byte: round to nearest, ties to even, finite
 * overflow saturated to +-448, sign of zero kept, NaN -> 0x7F | sign. */
uint8_t oracle_f32_to_e4m3(float f);
/* Element-wise array forms of the four conversions above (for the tests). */
void oracle_bf16_to_f32_n(int64_t n, const uint16_t *in, float *out);
void oracle_f32_to_bf16_n(int64_t n, const float *in, uint16_t *out);
void oracle_e4m3_to_f32_n(int64_t n, const uint8_t *in, float *out);
void oracle_f32_to_e4m3_n(int64_t n, const float *in, uint8_t *out);

/* ---- plan ---------------------------------------------------------------- */
/* Counts, per-rank offsets, stable slots and return addresses.  T may be 0
 * (an empty batch: every count and offset is 0).
 * Returns ORACLE_OK, ORACLE_BAD_EXPERT (nothing written) or ORACLE_CAPACITY
 * (counts/offsets written, slot_of written, src_of written only below cap). */
int oracle_plan(int R, int T, int E, int K, int cap, const int32_t *topk_idx,
                int32_t *expert_num_tokens, int32_t *expert_rank_offsets,
                int32_t *slot_of, int32_t *src_of);

/* Plan with ragged ranks and masked routing.  Entry (g, k) of token
 * g = r*T + t is routed iff t < clamp(num_tokens[r], 0, T) (num_tokens NULL:
 * every token) and topk_idx[g,k] != -1; entries of tokens beyond num_tokens
 * are ignored whatever they hold.  Counts, offsets and slots are those of
 * oracle_plan over the routed entries only; unrouted entries get
 * slot_of = -1.  A routed id outside [0, E) gives ORACLE_BAD_EXPERT. */
int oracle_plan_masked(int R, int T, int E, int K, int cap, const int32_t *topk_idx,
                       const int32_t *num_tokens, int32_t *expert_num_tokens,
                       int32_t *expert_rank_offsets, int32_t *slot_of, int32_t *src_of);

/* ---- dispatch ------------------------------------------------------------ */
/* bf16 payload: expert_x[e][slot_of[g,k]][:] = x[g][:] bit for bit. */
void oracle_dispatch_bf16(int N, int H, int E, int K, int cap,
                          const uint16_t *x, const int32_t *topk_idx,
                          const int32_t *slot_of, uint16_t *expert_x);

/* Quantise one H-element bf16 row to e4m3 with one fp32 scale per
 * 128-element block.  H must be a multiple of 128. */
void oracle_quant_row_e4m3(int H, const uint16_t *row, uint8_t *q,
                           float *scale);

/* fp8 payload: the quantised row of x[g] and its scales written to every
 * (expert, slot) the token goes to. */
void oracle_dispatch_fp8(int N, int H, int E, int K, int cap,
                         const uint16_t *x, const int32_t *topk_idx,
                         const int32_t *slot_of, uint8_t *expert_x,
                         float *expert_x_scale);

/* ---- combine ------------------------------------------------------------- */
/* y[g][h] = bf16( fp32 fma chain over k = 0..K-1 of
 *                 w[g,k] * expert_y[topk_idx[g,k]][slot_of[g,k]][h] ). */
void oracle_combine(int N, int H, int E, int K, int cap,
                    const uint16_t *expert_y, const int32_t *topk_idx,
                    const int32_t *slot_of, const float *topk_weights,
                    uint16_t *y);

/* Combine fused with the shared expert: as oracle_combine, but the fp32
 * accumulator starts at the shared expert's output for the token:
 * y[g][h] = bf16( fma chain over k of w*expert_y, starting from
 *                 float(shared[g][h]) ). */
void oracle_combine_shared(int N, int H, int E, int K, int cap,
                           const uint16_t *expert_y, const int32_t *topk_idx,
                           const int32_t *slot_of, const float *topk_weights,
                           const uint16_t *shared, uint16_t *y);

/* Router: for each of N tokens, the K largest of its E logits (ties: lower
 * expert index first), in that order, and their softmax weights computed in
 * fp64 from the largest logit and rounded once to fp32.  K <= E. */
void oracle_router_topk(int N, int E, int K, const float *logits, int32_t *topk_idx,
                        float *topk_weights);

/* e^x in binary32 by the algorithm this library fixes for SiLU (Cody-Waite
 * reduction with a two-part ln 2, degree-7 Taylor polynomial in Horner form
 * with fused multiply-adds, exact scaling by 2^n): +inf above 88.72, 0 below
 * -87.33. */
float oracle_exp_f32(float x);
/* SiLU(g) = g / (1 + e^-g) with oracle_exp_f32, in binary32. */
float oracle_silu_f32(float g);

/* Activation between the expert GEMMs: for expert e and row s <
 * clamp(expert_num_tokens[e], 0, cap), a = SiLU(gate) * up with gate, up the
 * two halves of expert_h[e][s] ([E, cap, 2I] bf16), then a 1x128 E4M3
 * quantisation of a exactly like oracle_quant_row_e4m3 (on fp32 values).
 * Writes act_q[E, cap, I] and act_scale[E, cap, I/128] for those rows only. */
void oracle_silu_mul_quant(int E, int cap, int I, const uint16_t *expert_h,
                           const int32_t *expert_num_tokens, uint8_t *act_q,
                           float *act_scale);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
