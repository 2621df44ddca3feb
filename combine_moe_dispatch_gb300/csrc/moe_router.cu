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
// lane looks for its next best (in calls bound by latency, each lane keeps
// its second-best ready as well: router_ff_kernel's TOP2).
//   The weights are computed in float-float (pairs of fp32 values) rather
// than fp64: this GPU's fp64 rate is a small fraction of its fp32 rate, and
// the fp64 softmax cost 0.7 us of the 4.5 us call at DeepSeek-V3 decode.
// The float-float result is within about 2^-36 of the exact weight before
// its one rounding to fp32, so it is the exactly rounded weight or a
// neighbour of it (tests/router_ff_check.c restates these steps on the CPU
// and checks them against fp64).
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
// 2^(j/32), j = 0..31, each as a float-float (hi, lo): hi = RN(2^(j/32)),
// lo = RN(2^(j/32) - hi), from the exact values (so within 2^-48 of them).
__device__ const float2 g_exp2_32[32] = {
    {0x1p+0f, 0x0p+0f}, {0x1.059b0ep+0f, -0x1.9d4f52p-25f}, {0x1.0b5586p+0f, 0x1.9f3122p-25f},
    {0x1.11301ep+0f, -0x1.fdb496p-25f}, {0x1.172b84p+0f, -0x1.c15742p-27f}, {0x1.1d4874p+0f, -0x1.d2e8cap-25f},
    {0x1.2387a6p+0f, 0x1.ceac48p-25f}, {0x1.29e9e0p+0f, -0x1.5c0424p-25f}, {0x1.306fe0p+0f, 0x1.4636e2p-25f},
    {0x1.371a74p+0f, -0x1.18aac6p-25f}, {0x1.3dea64p+0f, 0x1.824684p-25f}, {0x1.44e086p+0f, 0x1.8624b4p-30f},
    {0x1.4bfdaep+0f, -0x1.593abcp-25f}, {0x1.5342b6p+0f, -0x1.2c5610p-25f}, {0x1.5ab07ep+0f, -0x1.5bd5ecp-27f},
    {0x1.6247ecp+0f, -0x1.f8b550p-25f}, {0x1.6a09e6p+0f, 0x1.9fcef4p-26f}, {0x1.71f75ep+0f, 0x1.1d8beep-25f},
    {0x1.7a1148p+0f, -0x1.829fd0p-25f}, {0x1.82589ap+0f, -0x1.accc7cp-26f}, {0x1.8ace54p+0f, 0x1.15506ep-27f},
    {0x1.93737cp+0f, -0x1.e64744p-25f}, {0x1.9c4918p+0f, 0x1.51f848p-27f}, {0x1.a5503cp+0f, -0x1.b83b54p-25f},
    {0x1.ae89fap+0f, -0x1.a94b14p-26f}, {0x1.b7f770p+0f, -0x1.a09438p-25f}, {0x1.c199bep+0f, -0x1.3d56b2p-27f},
    {0x1.cb720ep+0f, -0x1.8837ccp-27f}, {0x1.d5818ep+0f, -0x1.822dbcp-27f}, {0x1.dfc974p+0f, -0x1.908c94p-25f},
    {0x1.ea4afap+0f, 0x1.52486cp-27f}, {0x1.f50766p+0f, -0x1.246eb0p-26f},
};

// e^d for d = dh + dl in [-64, 0] (dh + dl exact, |dl| <= ulp(dh) / 2), as a
// float-float with relative error about 2^-36 (the largest the CPU check of
// these steps finds over 3.8e7 arguments is 2^-36.35).  A table-driven form
// of Cody and Waite's reduction (Software Manual for the Elementary
// Functions, 1980; Tang, "Table-driven implementation of the exponential
// function in IEEE floating-point arithmetic", 1989): N = rint(32 d / ln 2)
// = 32 m + j, r = d - N ln2/32 with ln2/32 split as L1 + L2 + L3 (L1 has 12
// significant bits, so N L1 is exact for |N| < 4096, and dh - N L1 is exact
// by Sterbenz's lemma), |r| <= ln2/64 + 2^-16; then e^d = 2^m 2^(j/32) e^r,
// with e^r = 1 + r + r^2 (1/2 + r/6 + r^2/24 + r^3/120) (truncation below
// 2^-48), the part after r in float and the two additions in float-float.
// Lane i holds entry i of the table in (my_th, my_tl); every lane of the
// warp calls this together (the entry is fetched by shuffle).
__device__ __forceinline__ FF ff_exp_neg(float dh, float dl, float my_th, float my_tl) {
  const float kInv = 0x1.715476p+5f;                                 // 32 / ln 2
  const float kL1 = 0x1.62ep-6f, kL2 = 0x1.0bfbe8p-20f, kL3 = 0x1.cf79acp-45f;
  const float n = rintf(__fmul_rn(dh, kInv));                        // N in [-2955, 0]
  const int ni = (int)n;
  const int j = ni & 31, m = ni >> 5;                                // N = 32 m + j
  const float th = __shfl_sync(kAll, my_th, j), tl = __shfl_sync(kAll, my_tl, j);
  const float r1 = __fsub_rn(dh, __fmul_rn(n, kL1));                 // exact
  const float p2 = __fmul_rn(n, kL2);
  const float p2e = __fmaf_rn(n, kL2, -p2);                          // N L2 = p2 + p2e
  const FF s = two_sum(r1, -p2);
  const float low = __fsub_rn(__fadd_rn(__fsub_rn(s.l, p2e), dl), __fmul_rn(n, kL3));
  const FF r = fast_two_sum(s.h, low);
  float q = __fmaf_rn(r.h, 0x1.111112p-7f, 0x1.555556p-5f);          // 1/24 + r/120
  q = __fmaf_rn(q, r.h, 0x1.555556p-3f);                             // 1/6 + ...
  q = __fmaf_rn(q, r.h, 0.5f);                                       // 1/2 + ...
  const float pr = __fmul_rn(__fmul_rn(r.h, r.h), q);                // r^2 (1/2 + ...)
  const FF t = ff_add({1.0f, 0.0f}, ff_add(r, {pr, 0.0f}));          // e^r
  const FF u = ff_mul(t, {th, tl});
  const float two_m = __int_as_float((127 + m) << 23);               // 2^m, m in [-93, 0]
  return {__fmul_rn(u.h, two_m), __fmul_rn(u.l, two_m)};
}

// One warp per token (the steps are in the header comment).
//   Selection: each lane keeps its best (value, then lowest index) among its
//   remaining logits; a round is one warp maximum of the lanes' bests, a
//   ballot of the lanes holding it, and the lowest such lane gives up its
//   best.
//   TOP2 (for calls with at most one token per warp of one block per SM,
//   which latency bounds): each lane keeps its second-best ready too, so
//   the winner's next best is a select and the next round's maximum waits
//   for nothing more; every lane then searches its second-best again while
//   that maximum is in flight.  Otherwise only the winning lane searches,
//   after the round: fewer instructions, for calls bound by instruction
//   issue (Kimi-K2 decode: 7.26 against 10.05 us with TOP2).
//   Softmax: d_k = l_k - l_max is exact as a float-float (TwoSum); e^d_k
//   from ff_exp_neg (d_k < -64, -inf or NaN: in fp64, as the oracle does);
//   the sum of the K exponentials as a float-float butterfly; the quotient
//   q = RN(e_h y), y ~ 1/S_h, corrected once by the exact remainder e - q S,
//   and rounded once.  The result is within about 2^-36 of the exact weight
//   before that last rounding, so it is the exactly rounded weight or its
//   neighbour.
template <int VPL, bool TOP2>
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
  const float2 my_t = g_exp2_32[lane];          // constants: loaded before the wait
  pdl_wait_for_previous();
  for (int64_t g = w0; g < p.N; g += nw) {
    const float *row = p.logits + g * E;
    uint32_t key[VPL];
    if (vec) {
#pragma unroll
      for (int j = 0; j < VPL; j += 4) {
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(row + e0 + j));
        key[j] = TOP2 ? max(order_key(v.x), 1u) : order_key(v.x);
        key[j + 1] = TOP2 ? max(order_key(v.y), 1u) : order_key(v.y);
        key[j + 2] = TOP2 ? max(order_key(v.z), 1u) : order_key(v.z);
        key[j + 3] = TOP2 ? max(order_key(v.w), 1u) : order_key(v.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const uint32_t k = e0 + j < E ? order_key(__ldcs(row + e0 + j)) : 0u;
        key[j] = TOP2 && e0 + j < E ? max(k, 1u) : k;
      }
    }
    // Key 0 marks no logit, so a logit's key is at least 1 (only the NaN
    // with every bit set has key 0).  The two forms of that rule are the
    // same; each variant takes the one that measured faster for it (TOP2 at
    // DeepSeek-V3 decode 2.91 against 3.00 us; the other at Kimi-K2 decode
    // 7.01 against 7.7 us).
    if (!TOP2) {
#pragma unroll
      for (int j = 0; j < VPL; ++j) key[j] = key[j] ? key[j] : (e0 + j < E ? 1u : 0u);
    }
    // the best key among the lane's, leaving out index ex (VPL: none)
    auto best = [&](int ex, uint32_t &bk, int &bj) {
      uint32_t tk[VPL];
      int tj[VPL];
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        tk[j] = j == ex ? 0u : key[j];
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
    uint32_t b1k, b2k = 0;
    int b1j, b2j = 0;
    best(VPL, b1k, b1j);
    if (TOP2) best(b1j, b2k, b2j);
    float my_v = 0.0f;
    int my_e = 0;
    for (int k = 0; k < K; ++k) {
      const uint32_t top = __reduce_max_sync(kAll, b1k);
      const int w = __ffs(__ballot_sync(kAll, b1k == top)) - 1;
      const int e = __shfl_sync(kAll, e0 + b1j, w);
      if (lane == k) {
        my_v = key_value(top);
        my_e = e;
      }
      if (TOP2) {
        // no branch: every lane selects, so the next maximum can issue
        // before the second-best search below
        const bool win = lane == w;
#pragma unroll
        for (int j = 0; j < VPL; ++j) key[j] = (win && j == b1j) ? 0u : key[j];
        b1k = win ? b2k : b1k;
        b1j = win ? b2j : b1j;
        best(b1j, b2k, b2j);
      } else if (lane == w) {
#pragma unroll
        for (int j = 0; j < VPL; ++j)
          if (j == b1j) key[j] = 0u;
        best(VPL, b1k, b1j);
      }
    }
    // softmax over the K chosen logits; lane 0 holds the largest.  Every
    // lane runs the float-float exponential (it fetches its table entry by
    // shuffle); lanes past K, and lanes whose difference is below -64, -inf
    // or NaN, run it on 0 and drop the result.
    const float m = __shfl_sync(kAll, my_v, 0);
    const FF d = two_sum(my_v, -m);
    const bool fast = lane < K && d.h >= -64.0f;
    FF ek = ff_exp_neg(fast ? d.h : 0.0f, fast ? d.l : 0.0f, my_t.x, my_t.y);
    double z = 0.0;
    const bool slow = lane < K && !fast;
    if (slow) {                                  // tiny, -inf or NaN: fp64
      z = exp((double)my_v - (double)m);
      ek.h = (float)z;
      ek.l = (float)(z - (double)ek.h);
    }
    if (lane >= K) ek = {0.0f, 0.0f};
    FF sum = ek;
    for (int l = 0; l < lg; ++l) {
      const FF o = {__shfl_xor_sync(kAll, sum.h, 1 << l), __shfl_xor_sync(kAll, sum.l, 1 << l)};
      sum = ff_add(sum, o);
    }
    if (lane < K) {
      float wk;
      if (!slow) {
        // y ~ 1/S_h from the approximate reciprocal (S_h in [1, 32]); the
        // remainder correction makes the result the same for any y within
        // 2 ulps of 1/S_h (the CPU check runs y = RN(1/S_h) moved by -2..2
        // ulps)
        float y;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(sum.h));
        const float q = __fmul_rn(ek.h, y);
        const float pr = __fmul_rn(q, sum.h);
        const float pe = __fmaf_rn(q, sum.h, -pr);            // q S_h = pr + pe
        const float rem = __fadd_rn(__fsub_rn(__fsub_rn(ek.h, pr), pe),
                                    __fsub_rn(ek.l, __fmul_rn(q, sum.l)));
        wk = __fadd_rn(q, __fmul_rn(rem, y));
      } else {
        wk = (float)(z / ((double)sum.h + (double)sum.l));
      }
      p.topk_idx[g * K + lane] = my_e;
      p.topk_weights[g * K + lane] = wk;
    }
  }
}

namespace {
template <int VPL, bool TOP2>
cudaError_t launch_vpl2(const RouterParams &p, cudaStream_t stream) {
  const int grid = persistent_grid((const void *)router_ff_kernel<VPL, TOP2>, kRouterThreads, p.N);
  return launch_after_previous(router_ff_kernel<VPL, TOP2>, grid, kRouterThreads, p, stream);
}
// TOP2 when every token gets a warp of a single block per SM: the call is
// then one token's latency (DeepSeek-V3 decode, 1024 tokens: 3.14 against
// 3.18 us without).
template <int VPL>
cudaError_t launch_vpl(const RouterParams &p, cudaStream_t stream) {
  const int64_t one_round = (int64_t)device_sm_count() * (kRouterThreads / 32);
  return p.N <= one_round ? launch_vpl2<VPL, true>(p, stream) : launch_vpl2<VPL, false>(p, stream);
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
