// moe_router.cu -- top-K expert selection and routing weights from router logits.
//
// What it computes ("Efficient and portable mixture-of-experts
// communication", Introduction; "Lower latency and higher throughput with
// multi-node DeepSeek deployment", MoE Router): for every token, the K
// experts with the largest logits, in descending order (ties: lower expert
// index first), and weights = softmax over those K logits, exp(l_k - l_max)
// / sum in fp64, rounded once to fp32.  The indices feed moe_plan directly.
//
// How: one warp per token, a block's 8 warps on 8 consecutive tokens.  The E
// logits are spread over the lanes in registers (coalesced loads); K rounds
// of a warp-wide arg-max each remove one expert: each lane's best (value,
// then lowest index) among its logits, then two warp reductions, the
// largest order-preserving key and the lowest expert holding it.  The
// chosen logits of the block's tokens then go to shared memory, where one
// thread per value computes its exponential and one thread per token adds
// its token's K exponentials in ascending k (a sequential sum, so the result
// does not depend on a reduction tree); one thread per value divides and
// stores, so the outputs of the block are written as one coalesced run.
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
// The float of a key (+0 for a key of zero).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int VPL>
__global__ void __launch_bounds__(kRouterThreads)
router_kernel(RouterParams p) {
  constexpr int kWarps = kRouterThreads / 32;
  // the block's tokens' chosen logits minus their maximum, exponentials and
  // ids, [warp][k]; K <= 32, so kWarps * K <= kRouterThreads
  __shared__ double s_d[kWarps * kMaxTopK];
  __shared__ double s_sum[kWarps];
  __shared__ int32_t s_e[kWarps * kMaxTopK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int K = p.K;
  pdl_wait_for_previous();
  // One token per warp; the block's kWarps tokens are consecutive, and every
  // warp runs every iteration (the barriers), idle past the last token.
  for (int64_t base = (int64_t)blockIdx.x * kWarps; base < p.N; base += (int64_t)gridDim.x * kWarps) {
    const int64_t g = base + warp;
    const bool live = g < p.N;
    float v[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = j * 32 + lane;
      v[j] = (live && e < p.E) ? __ldcs(p.logits + g * p.E + e) : -INFINITY;
    }
    uint32_t taken = 0;
    float my_v = 0.0f;
    int my_e = 0;
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int be = INT32_MAX;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = j * 32 + lane;
        const bool cand = e < p.E && !((taken >> j) & 1u);
        if (cand && (v[j] > bv || (v[j] == bv && e < be))) {
          bv = v[j];
          be = e;
        }
      }
      // the warp's best: the largest key, then the lowest expert holding it
      const uint32_t key = order_key(bv);
      const uint32_t top = __reduce_max_sync(kAll, key);
      const uint32_t win = __reduce_min_sync(kAll, key == top ? (uint32_t)be : 0xFFFFFFFFu);
      be = (int)win;
      if (be != INT32_MAX && (be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == k) {
        my_v = key_value(top);
        my_e = be;
      }
    }
    // The fp64 part runs once per value, not once per warp and token: this
    // GPU's fp64 rate is low, and a warp-wide fp64 instruction costs the
    // same with K lanes active as with 32.
    const float m = __shfl_sync(kAll, my_v, 0);
    if (lane < K) {
      s_d[warp * K + lane] = (double)my_v - (double)m;
      s_e[warp * K + lane] = my_e;
    }
    __syncthreads();
    const int nv = kWarps * K;                     // values of the block's tokens
    if (tid < nv) s_d[tid] = exp(s_d[tid]);
    __syncthreads();
    if (tid < kWarps) {                            // the sum in ascending k, as a sequential sum
      double sum = 0.0;
      for (int k = 0; k < K; ++k) sum += s_d[tid * K + k];
      s_sum[tid] = sum;
    }
    __syncthreads();
    if (tid < nv && base + tid / K < p.N) {        // consecutive outputs: coalesced
      p.topk_idx[base * K + tid] = s_e[tid];
      p.topk_weights[base * K + tid] = (float)(s_d[tid] / s_sum[tid / K]);
    }
    __syncthreads();
  }
}

namespace {
template <int VPL>
cudaError_t launch_vpl(const RouterParams &p, cudaStream_t stream) {
  const int grid = persistent_grid((const void *)router_kernel<VPL>, kRouterThreads, p.N);
  return launch_after_previous(router_kernel<VPL>, grid, kRouterThreads, p, stream);
}
}  // namespace

cudaError_t launch_router(const RouterParams &p, cudaStream_t stream) {
  const int need = (p.E + 31) / 32;
  if (need <= 1) return launch_vpl<1>(p, stream);
  if (need <= 2) return launch_vpl<2>(p, stream);
  if (need <= 4) return launch_vpl<4>(p, stream);
  if (need <= 8) return launch_vpl<8>(p, stream);
  if (need <= 16) return launch_vpl<16>(p, stream);
  return launch_vpl<32>(p, stream);
}

}  // namespace moe
