// moe_router.cu -- top-K expert selection and routing weights from router logits.
//
// What it computes ("Efficient and portable mixture-of-experts
// communication", Introduction; "Lower latency and higher throughput with
// multi-node DeepSeek deployment", MoE Router): for every token, the K
// experts with the largest logits, in descending order (ties: lower expert
// index first), and weights = softmax over those K logits, exp(l_k - l_max)
// / sum in fp64, rounded once to fp32.  The indices feed moe_plan directly.
//
// How: one warp per token.  The E logits are spread over the lanes in
// registers (coalesced loads); K rounds of a warp-wide arg-max (value, then
// index) each remove one expert.  Lanes 0..K-1 keep the chosen (logit,
// expert); every lane adds the K exponentials in ascending k, the same order
// as a sequential sum, so the result does not depend on a reduction tree.
#include <math.h>
#include <stdint.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kRouterThreads = 256;
constexpr unsigned kAll = 0xFFFFFFFFu;

template <int VPL>
__global__ void __launch_bounds__(kRouterThreads)
router_kernel(RouterParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kRouterThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kRouterThreads) >> 5;
  pdl_wait_for_previous();
  for (int64_t g = warp0; g < p.N; g += nwarps) {
    const float *row = p.logits + g * p.E;
    float v[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = j * 32 + lane;
      v[j] = e < p.E ? __ldcs(row + e) : -INFINITY;
    }
    uint32_t taken = 0;
    float my_v = 0.0f;
    int my_e = 0;
    for (int k = 0; k < p.K; ++k) {
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
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(kAll, bv, off);
        const int oe = __shfl_xor_sync(kAll, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if (be != INT32_MAX && (be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == k) {
        my_v = bv;
        my_e = be;
      }
    }
    const double m = __shfl_sync(kAll, (double)my_v, 0);
    const double z = lane < p.K ? exp((double)my_v - m) : 0.0;
    double sum = 0.0;
    for (int k = 0; k < p.K; ++k) sum += __shfl_sync(kAll, z, k);
    if (lane < p.K) {
      p.topk_idx[g * p.K + lane] = my_e;
      p.topk_weights[g * p.K + lane] = (float)(z / sum);
    }
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
