// moe_combine.cu -- gather-weighted-reduce of expert outputs back to tokens.
//
// What it computes ("Efficient and portable mixture-of-experts
// communication", Introduction and Combine; "Enabling trillion-parameter
// models on AWS EFA", Dispatch and Combine):
//   y[g][h] = bf16_rn( acc ),  acc = 0; for k = 0..K-1:
//             acc = fma(w[g,k], float(expert_y[idx[g,k]][slot_of[g,k]][h]), acc)
// i.e. the receiver-side weighted sum of the 16-bit expert outputs, one fp32
// accumulator per element, fixed k order, one final rounding.  With a
// shared-expert output ("Lower latency and higher throughput with
// multi-node DeepSeek deployment", Expert Parallelism) the accumulator
// starts from it instead of +0, which saves a separate read-add-write pass.
//
// How: a warp takes one (token, segment) task at a time; lanes 0..K-1 hold
// the token's K (expert, slot, weight) and broadcast them by shuffle.  For a
// group of KG experts the warp issues all KG x U 16-byte loads before the
// first multiply-add, so each lane keeps KG*U*16 bytes of reads in flight
// (256 B per lane, 8 KB per warp, 16 warps per SM for K = 8; measured
// faster than 128 B per lane at 32 warps per SM); only populated rows are
// read.  The
// accumulators stay in registers and the bf16 result is stored once, 16
// bytes per lane.
#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kCombineThreads = 256;

constexpr unsigned kFullMask = 0xFFFFFFFFu;

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4 &v) {
  const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fmaf_rn(w, __uint_as_float(a[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(a[i] & 0xFFFF0000u), acc[2 * i + 1]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

// Loads in flight per lane are KG * U * 16 bytes; MINB resident blocks per SM
// set the register budget (64 registers at 4, 85 at 3, 128 at 2).
template <int KG, int U, int MINB>
__global__ void __launch_bounds__(kCombineThreads, MINB)
combine_kernel(CombineParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kCombineThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kCombineThreads) >> 5;
  const int cpr = p.H / 8;           // 16-byte chunks per row
  constexpr int cpt = 32 * U;        // chunks per task
  const int tpr = (cpr + cpt - 1) / cpt;
  const int64_t ntasks = (int64_t)p.N * tpr;
  TaskCursor cur(warp0, nwarps, tpr);
  // After the wait, thread 0 reads the status word while every warp's first
  // routing loads are in flight (before, one round trip after the other:
  // 22.1 -> 21.9 us at DeepSeek-V3 decode, 18.5 -> 18.1 us at the
  // Mixtral-shaped layer).
  __shared__ int32_t s_status;
  pdl_wait_for_previous();
  if (threadIdx.x == 0) s_status = read_status(p.hdr);
  int e_l = -1, s_l = -1;
  float w_l = 0.0f;
  if (warp0 < ntasks && lane < p.K) {
    e_l = __ldg(p.topk_idx + (int64_t)cur.g * p.K + lane);
    s_l = __ldg(p.slot_of + (int64_t)cur.g * p.K + lane);
    w_l = __ldg(p.topk_weights + (int64_t)cur.g * p.K + lane);
  }
  __syncthreads();
  if (s_status != MOE_OK || warp0 >= ntasks) return;
  // The routing of a warp's next task is loaded while the current task's
  // rows are read, so each task waits for one memory round trip (its rows),
  // not two (its routing, then its rows).
  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int64_t g = cur.g;
    const int seg = cur.seg;
    // slot -1: an entry the plan did not route (skipped; a token with no
    // routed entry gets y = +0).  Other out-of-range entries are reported.
    const bool routed = lane < p.K && s_l != -1;
    const bool e_ok = e_l >= 0 && e_l < p.E;
    const bool ok = routed && e_ok && s_l >= 0 && s_l < p.cap;
    if (seg == 0 && routed && !ok)
      report_status(p.hdr, e_ok ? MOE_ERR_CAPACITY : MOE_ERR_BAD_EXPERT);
    const unsigned okmask = __ballot_sync(kFullMask, ok);
    const int ce_l = e_l, cs_l = s_l;
    const float cw_l = w_l;
    cur = cur.next();
    const bool more = task + nwarps < ntasks;

    const int c0 = seg * cpt + lane;
    float acc[U][8];
    if (p.shared) {                       // the shared expert's output seeds the accumulator
      const uint16_t *srow = p.shared + g * p.H;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32;
        const uint4 v = c < cpr ? __ldcs(reinterpret_cast<const uint4 *>(srow + (int64_t)c * 8))
                                : make_uint4(0, 0, 0, 0);
        const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[u][2 * i] = __uint_as_float(a[i] << 16);
          acc[u][2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
    }

    for (int kb = 0; kb < p.K; kb += KG) {
      uint4 v[KG][U];
#pragma unroll
      for (int kk = 0; kk < KG; ++kk) {
        const int k = kb + kk;
        const int e = __shfl_sync(kFullMask, ce_l, k & 31);
        const int s = __shfl_sync(kFullMask, cs_l, k & 31);
        const bool use = k < p.K && ((okmask >> (k & 31)) & 1u);
        const uint16_t *row = p.expert_y + ((int64_t)(use ? e : 0) * p.cap + (use ? s : 0)) * p.H;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + u * 32;
          v[kk][u] = (use && c < cpr) ? __ldcs(reinterpret_cast<const uint4 *>(row + (int64_t)c * 8))
                                      : make_uint4(0, 0, 0, 0);
        }
      }
      if (kb == 0 && more && lane < p.K) {   // the next task's routing, behind this task's first rows
        e_l = __ldg(p.topk_idx + (int64_t)cur.g * p.K + lane);
        s_l = __ldg(p.slot_of + (int64_t)cur.g * p.K + lane);
        w_l = __ldg(p.topk_weights + (int64_t)cur.g * p.K + lane);
      }
#pragma unroll
      for (int kk = 0; kk < KG; ++kk) {
        const int k = kb + kk;
        const float w = __shfl_sync(kFullMask, cw_l, k & 31);
        if (k < p.K && ((okmask >> (k & 31)) & 1u)) {
#pragma unroll
          for (int u = 0; u < U; ++u) fma8(acc[u], w, v[kk][u]);
        }
      }
    }

    uint16_t *out = p.y + g * p.H;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c < cpr) {
        uint4 o;
        o.x = pack_bf16x2(acc[u][0], acc[u][1]);
        o.y = pack_bf16x2(acc[u][2], acc[u][3]);
        o.z = pack_bf16x2(acc[u][4], acc[u][5]);
        o.w = pack_bf16x2(acc[u][6], acc[u][7]);
        *reinterpret_cast<uint4 *>(out + (int64_t)c * 8) = o;
      }
    }
  }
}

#ifndef MOE_COMBINE_U8
#define MOE_COMBINE_U8 2   // chunks per lane for K > 4: 16 loads (256 B) in flight per lane
#endif

namespace {
template <int KG, int U, int MINB>
cudaError_t launch_variant(const CombineParams &p, cudaStream_t stream) {
  const int cpr = p.H / 8;
  const int64_t tasks = (int64_t)p.N * ((cpr + 32 * U - 1) / (32 * U));
  const int grid =
      persistent_grid((const void *)combine_kernel<KG, U, MINB>, kCombineThreads, tasks);
  return launch_after_previous(combine_kernel<KG, U, MINB>, grid, kCombineThreads, p, stream);
}
}  // namespace

// Chunks per lane and resident blocks per SM, by K.  Measured (graphs of
// back-to-back launches over rotating buffer sets): Mixtral (K = 2) 2 chunks
// at 4 blocks 18.5 us, 4 at 3 18.7, 4 at 2 20.2, 1 at 8 19.8; DeepSeek-V3
// decode (K = 8) 2 at 2 21.4 us, 1 at 4 23.4, 2 at 3 29.5.
#ifndef MOE_COMBINE_U2
#define MOE_COMBINE_U2 2
#endif
#ifndef MOE_COMBINE_MINB2
#define MOE_COMBINE_MINB2 4
#endif
#ifndef MOE_COMBINE_MINB8
#define MOE_COMBINE_MINB8 (MOE_COMBINE_U8 == 1 ? 4 : 2)
#endif

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
  if (p.K <= 2) return launch_variant<2, MOE_COMBINE_U2, MOE_COMBINE_MINB2>(p, stream);
  if (p.K <= 4) return launch_variant<4, 2, 3>(p, stream);
  return launch_variant<8, MOE_COMBINE_U8, MOE_COMBINE_MINB8>(p, stream);
}

}  // namespace moe
