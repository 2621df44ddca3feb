// moe_router.cu -- top-K expert selection and routing weights from router logits.
//
// What it computes ("Efficient and portable mixture-of-experts
// communication", Introduction; "Lower latency and higher throughput with
// multi-node DeepSeek deployment", MoE Router): for every token, the K
// experts with the largest logits, in descending order (ties: lower expert
// index first), and weights = softmax over those K logits, exp(l_k - l_max)
// / sum, rounded once to fp32.  The indices feed moe_plan directly.
//
// How: one warp per token.  Lane j holds the logits of experts
// [j*VPL, (j+1)*VPL) in registers (16-byte loads when the lanes are full), so
// that among lanes holding the same largest value the lowest lane holds the
// lowest expert.  Each lane keeps its best remaining logit (value, then
// lowest index); K rounds of a warp maximum over the lanes' bests and a
// ballot of the lanes that hold it pick the experts, and only the winning
// lane looks for its next best.
//   The weights are computed in float-float (pairs of fp32 values) rather
// than fp64: this GPU's fp64 rate is a small fraction of its fp32 rate, and
// the fp64 softmax cost 0.7 us of the 4.5 us call at DeepSeek-V3 decode.
// The float-float result is within 2^-34 of the exact weight before its one
// rounding to fp32, so it is the exactly rounded weight or a neighbour of
// it (tests/router_ff_check.c restates these steps on the CPU and checks
// them against fp64).
#include <math.h>
#include <stdint.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kRouterThreads = 256;
constexpr unsigned kAll = 0xFFFFFFFFu;

// An unsigned key whose order is the order of the floats: the sign bit set
// for non-negative values, all bits flipped for negative ones, with -0
// mapped to +0 (the two compare equal).  NaN logits are unspecified.
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// The float of a key (never called on 0, the key that marks no logit).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// --- float-float arithmetic (Dekker 1971; Knuth, TAOCP vol. 2, 4.2.2) ---
// A value is an unevaluated sum hi + lo.  Every operation is an explicit
// round-to-nearest intrinsic, so the compiler cannot contract or reorder it.
struct FF {
  float h, l;
};
// a + b = s + e exactly (Knuth's TwoSum; no ordering of |a|, |b| needed)
__device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
// a + b = s + e exactly when |a| >= |b| (Dekker's Fast2Sum)
__device__ __forceinline__ FF fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
// Sum of two float-floats.  The low parts are added first, which keeps the
// operation commutative (so every lane of a butterfly gets the same sum).
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const FF s = two_sum(a.h, b.h);
  return fast_two_sum(s.h, __fadd_rn(s.l, __fadd_rn(a.l, b.l)));
}
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const float p = __fmul_rn(a.h, b.h);
  float e = __fmaf_rn(a.h, b.h, -p);           // a.h * b.h = p + e exactly
  e = __fmaf_rn(a.h, b.l, __fmaf_rn(a.l, b.h, e));
  return fast_two_sum(p, e);
}
// c + r * t for a float c exactly representable (1, 1/2)
__device__ __forceinline__ FF ff_horner(float c, FF r, FF t) {
  return ff_add({c, 0.0f}, ff_mul(r, t));
}

// e^d for d = dh + dl in [-64, 0] (dh + dl exact, |dl| <= ulp(dh) / 2), as a
// float-float with relative error about 2^-34 (the largest the CPU check of
// these steps finds over 3.8e7 arguments).  Cody and Waite's reduction
// (Software Manual for the Elementary Functions, 1980): n = rint(d / ln 2),
// r = d - n ln 2 with ln 2 split as L1 + L2 + L3 (L1 has 15 significant bits,
// so n L1 is exact for |n| < 512, and dh - n L1 is exact by Sterbenz's
// lemma); then the Taylor series of e^r to r^9 / 9! (truncation below
// 2^-37 for |r| <= ln 2 / 2 + 2^-16), its low-order part
// 1 + r + r^2/2 + r^3 (1/6 + r Q(r)) in float-float, Q in float; e^d = 2^n e^r.
__device__ __forceinline__ FF ff_exp_neg(float dh, float dl) {
  const float kInvLn2 = 0x1.715476p+0f;
  const float kL1 = 0x1.62e4p-1f, kL2 = 0x1.7f7d1cp-20f, kL3 = 0x1.ef357ap-45f;
  const float n = rintf(__fmul_rn(dh, kInvLn2));
  const float r1 = __fsub_rn(dh, __fmul_rn(n, kL1));              // exact
  const float p2 = __fmul_rn(n, kL2);
  const float p2e = __fmaf_rn(n, kL2, -p2);                         // n L2 = p2 + p2e
  const FF s = two_sum(r1, -p2);
  const float low = __fsub_rn(__fadd_rn(__fsub_rn(s.l, p2e), dl), __fmul_rn(n, kL3));
  const FF r = fast_two_sum(s.h, low);
  // Q(r) = 1/4! + r/5! + ... + r^5/9!, in float
  float q = 0x1.71de3ap-19f;
  q = __fmaf_rn(q, r.h, 0x1.a01a02p-16f);
  q = __fmaf_rn(q, r.h, 0x1.a01a02p-13f);
  q = __fmaf_rn(q, r.h, 0x1.6c16c2p-10f);
  q = __fmaf_rn(q, r.h, 0x1.111112p-7f);
  q = __fmaf_rn(q, r.h, 0x1.555556p-5f);
  const float rqh = __fmul_rn(r.h, q);                               // r Q = rqh + rql
  const float rql = __fmaf_rn(r.l, q, __fmaf_rn(r.h, q, -rqh));
  FF t = ff_add({0x1.555556p-3f, -0x1.555556p-28f}, {rqh, rql});     // 1/6 + r Q
  t = ff_horner(0.5f, r, t);
  t = ff_horner(1.0f, r, t);
  t = ff_horner(1.0f, r, t);
  const float two_n = __int_as_float((127 + (int)n) << 23);        // 2^n, n in [-93, 0]
  return {__fmul_rn(t.h, two_n), __fmul_rn(t.l, two_n)};
}

// One warp per token (the steps are in the header comment).
//   Selection: each lane keeps its best (value, then lowest index) among its
//   remaining logits; a round is one warp maximum of the lanes' bests, a
//   ballot of the lanes holding it, and the lowest such lane gives up its
//   best and finds its next.
//   Softmax: d_k = l_k - l_max is exact as a float-float (TwoSum); e^d_k
//   from ff_exp_neg (d_k < -64, -inf or NaN: in fp64, as the oracle does);
//   the sum of the K exponentials as a float-float butterfly; the quotient
//   q = RN(e_h / S_h) corrected once by the remainder e - q S, and rounded
//   once.  The result is within 2^-34 of the exact weight before that last
//   rounding, so it is the exactly rounded weight or its neighbour.
template <int VPL>
__global__ void __launch_bounds__(kRouterThreads)
router_ff_kernel(RouterParams p) {
  const int lane = threadIdx.x & 31;
  const int K = p.K, E = p.E;
  const int e0 = lane * VPL;
  const int64_t w0 = ((int64_t)blockIdx.x * kRouterThreads + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * kRouterThreads) >> 5;
  const bool vec = (VPL % 4 == 0) && E == 32 * VPL && ((uintptr_t)p.logits & 15u) == 0;
  int lg = 1;                                   // butterfly levels: 2^lg >= K
  while ((1 << lg) < K) ++lg;
  pdl_wait_for_previous();
  for (int64_t g = w0; g < p.N; g += nw) {
    const float *row = p.logits + g * E;
    uint32_t key[VPL];
    if (vec) {
#pragma unroll
      for (int j = 0; j < VPL; j += 4) {
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(row + e0 + j));
        key[j] = order_key(v.x);
        key[j + 1] = order_key(v.y);
        key[j + 2] = order_key(v.z);
        key[j + 3] = order_key(v.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < VPL; ++j) key[j] = e0 + j < E ? order_key(__ldcs(row + e0 + j)) : 0u;
    }
#pragma unroll
    for (int j = 0; j < VPL; ++j) key[j] = key[j] ? key[j] : (e0 + j < E ? 1u : 0u);   // 0: none
    auto best = [&](uint32_t &bk, int &bj) {
      uint32_t tk[VPL];
      int tj[VPL];
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        tk[j] = key[j];
        tj[j] = j;
      }
#pragma unroll
      for (int st = 1; st < VPL; st <<= 1)
#pragma unroll
        for (int j = 0; j + st < VPL; j += 2 * st)
          if (tk[j + st] > tk[j]) {       // ties keep the lower index
            tk[j] = tk[j + st];
            tj[j] = tj[j + st];
          }
      bk = tk[0];
      bj = tj[0];
    };
    uint32_t bk;
    int bj;
    best(bk, bj);
    float my_v = 0.0f;
    int my_e = 0;
    for (int k = 0; k < K; ++k) {
      const uint32_t top = __reduce_max_sync(kAll, bk);
      const int w = __ffs(__ballot_sync(kAll, bk == top)) - 1;
      const int e = __shfl_sync(kAll, e0 + bj, w);
      if (lane == k) {
        my_v = key_value(top);
        my_e = e;
      }
      if (lane == w) {
#pragma unroll
        for (int j = 0; j < VPL; ++j)
          if (j == bj) key[j] = 0u;
        best(bk, bj);
      }
    }
    // softmax over the K chosen logits; lane 0 holds the largest
    const float m = __shfl_sync(kAll, my_v, 0);
    FF ek = {0.0f, 0.0f};
    double z = 0.0;
    bool slow = false;
    if (lane < K) {
      const FF d = two_sum(my_v, -m);
      if (d.h >= -64.0f) {
        ek = ff_exp_neg(d.h, d.l);
      } else {                                   // tiny, -inf or NaN: fp64
        slow = true;
        z = exp((double)my_v - (double)m);
        ek.h = (float)z;
        ek.l = (float)(z - (double)ek.h);
      }
    }
    FF sum = ek;
    for (int l = 0; l < lg; ++l) {
      const FF o = {__shfl_xor_sync(kAll, sum.h, 1 << l), __shfl_xor_sync(kAll, sum.l, 1 << l)};
      sum = ff_add(sum, o);
    }
    if (lane < K) {
      float wk;
      if (!slow) {
        const float q = __fdiv_rn(ek.h, sum.h);
        const float pr = __fmul_rn(q, sum.h);
        const float pe = __fmaf_rn(q, sum.h, -pr);
        const float rem = __fadd_rn(__fsub_rn(__fsub_rn(ek.h, pr), pe),
                                    __fsub_rn(ek.l, __fmul_rn(q, sum.l)));
        wk = __fadd_rn(q, __fdiv_rn(rem, sum.h));
      } else {
        wk = (float)(z / ((double)sum.h + (double)sum.l));
      }
      p.topk_idx[g * K + lane] = my_e;
      p.topk_weights[g * K + lane] = wk;
    }
  }
}

namespace {
template <int VPL>
cudaError_t launch_vpl(const RouterParams &p, cudaStream_t stream) {
  const int grid = persistent_grid((const void *)router_ff_kernel<VPL>, kRouterThreads, p.N);
  return launch_after_previous(router_ff_kernel<VPL>, grid, kRouterThreads, p, stream);
}
}  // namespace

cudaError_t launch_router(const RouterParams &p, cudaStream_t stream) {
  const int need = (p.E + 31) / 32;
  if (need <= 1) return launch_vpl<1>(p, stream);
  if (need <= 2) return launch_vpl<2>(p, stream);
  if (need <= 4) return launch_vpl<4>(p, stream);
  if (need <= 8) return launch_vpl<8>(p, stream);
  if (need <= 12) return launch_vpl<12>(p, stream);   // E = 384: full lanes, 16-byte loads
  if (need <= 16) return launch_vpl<16>(p, stream);
  return launch_vpl<32>(p, stream);
}

}  // namespace moe
