// moe_dispatch.cu -- row scatter of token activations into padded per-expert
// buffers, as a bf16 copy or fused with fp8 E4M3 1x128 block quantisation.
//
// What it computes ("Efficient and portable mixture-of-experts
// communication", Dispatch; "Lower latency and higher throughput with
// multi-node DeepSeek deployment", Quantization):
//   bf16:  expert_x[e][s][:] = x[g][:]            for every (g,k), e = idx, s = slot_of
//   fp8:   per 128-element block b of x[g]: scale = amax/448,
//          q = e4m3_rn_satfinite(x / scale) (all-zero block: scale 0, q 0);
//          the bytes and the H/128 scales go to every (e, s) of the token.
//
// How: work is cut by token, never by expert, so a skewed routing costs the
// same as a uniform one.  A warp takes one (token, 2048-element segment)
// task at a time from a grid sized to fill every SM: its lanes read the
// segment once with 16-byte loads (all loads issued before any store), then
// write it K times with coalesced 16-byte (bf16) or 8-byte (fp8) stores.  In
// the fp8 path each half-warp owns one 128-element block: the absmax is a
// 4-step butterfly over 16 lanes, and the block's scale is computed once and
// shared by all K copies.  The 16 scales of a segment are gathered into
// lanes 0..15 and stored as one 64-byte run per destination row.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kDispatchThreads = 256;
constexpr int kBf16ChunksPerLane = 8;   // 8 x 16 B per lane: a 2048-element segment
constexpr int kFp8PairsPerTask = 8;     // 8 x 256 elements: 16 blocks of 128
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}

// Routing of token g held by lanes 0..K-1; returns the mask of valid k and
// reports out-of-range entries once per token.
__device__ __forceinline__ unsigned load_routes(const DispatchParams &p, int64_t g, int lane,
                                                bool report, int &e_l, int &s_l) {
  e_l = -1;
  s_l = -1;
  if (lane < p.K) {
    e_l = __ldg(p.topk_idx + g * p.K + lane);
    s_l = __ldg(p.slot_of + g * p.K + lane);
  }
  const bool e_ok = e_l >= 0 && e_l < p.E;
  const bool ok = lane < p.K && e_ok && s_l >= 0 && s_l < p.cap;
  if (report && lane < p.K && !ok)
    report_status(p.hdr, e_ok ? MOE_ERR_CAPACITY : MOE_ERR_BAD_EXPERT);
  return __ballot_sync(kFull, ok);
}

__global__ void __launch_bounds__(kDispatchThreads)
dispatch_bf16_kernel(DispatchParams p) {
  __shared__ int32_t s_status;
  if (threadIdx.x == 0) s_status = read_status(p.hdr);
  __syncthreads();
  if (s_status != MOE_OK) return;

  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kDispatchThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDispatchThreads) >> 5;
  const int cpr = p.H / 8;                               // 16-byte chunks per row
  constexpr int cpt = 32 * kBf16ChunksPerLane;           // chunks per task
  const int tpr = (cpr + cpt - 1) / cpt;                 // tasks per row
  const int64_t ntasks = (int64_t)p.N * tpr;

  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int64_t g = task / tpr;
    const int seg = (int)(task - g * tpr);
    int e_l, s_l;
    const unsigned okmask = load_routes(p, g, lane, seg == 0, e_l, s_l);

    const uint16_t *src = p.x + g * p.H;
    const int c0 = seg * cpt + lane;
    uint4 v[kBf16ChunksPerLane];
#pragma unroll
    for (int u = 0; u < kBf16ChunksPerLane; ++u) {
      const int c = c0 + u * 32;
      v[u] = c < cpr ? ld_stream16(src + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
    }
    for (int k = 0; k < p.K; ++k) {
      const int e = __shfl_sync(kFull, e_l, k);
      const int s = __shfl_sync(kFull, s_l, k);
      if (!((okmask >> k) & 1u)) continue;
      uint16_t *dst = static_cast<uint16_t *>(p.expert_x) + ((int64_t)e * p.cap + s) * p.H;
#pragma unroll
      for (int u = 0; u < kBf16ChunksPerLane; ++u) {
        const int c = c0 + u * 32;
        if (c < cpr) *reinterpret_cast<uint4 *>(dst + (int64_t)c * 8) = v[u];
      }
    }
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> two E4M3 bytes (first in the low byte), nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__global__ void __launch_bounds__(kDispatchThreads)
dispatch_fp8_kernel(DispatchParams p) {
  __shared__ int32_t s_status;
  if (threadIdx.x == 0) s_status = read_status(p.hdr);
  __syncthreads();
  if (s_status != MOE_OK) return;

  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;     // which block of the 256-element pair
  const int sub = lane & 15;      // 8 elements (16 bytes in, 8 bytes out) per lane
  const int64_t warp0 = ((int64_t)blockIdx.x * kDispatchThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDispatchThreads) >> 5;
  const int nb = p.H / 128;                                  // blocks per row
  constexpr int bpt = 2 * kFp8PairsPerTask;                  // blocks per task (16)
  const int tpr = (nb + bpt - 1) / bpt;
  const int64_t ntasks = (int64_t)p.N * tpr;

  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int64_t g = task / tpr;
    const int seg = (int)(task - g * tpr);
    int e_l, s_l;
    const unsigned okmask = load_routes(p, g, lane, seg == 0, e_l, s_l);

    const uint16_t *src = p.x + g * p.H;
    uint4 v[kFp8PairsPerTask];
#pragma unroll
    for (int it = 0; it < kFp8PairsPerTask; ++it) {
      const int blk = seg * bpt + it * 2 + half;
      v[it] = blk < nb ? ld_stream16(src + (int64_t)blk * 128 + sub * 8) : make_uint4(0, 0, 0, 0);
    }

    uint2 q[kFp8PairsPerTask];
    float my_scale = 0.0f;   // lane L < 16 ends up with the scale of block seg*16 + L
#pragma unroll
    for (int it = 0; it < kFp8PairsPerTask; ++it) {
      const uint32_t w[4] = {v[it].x, v[it].y, v[it].z, v[it].w};
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
      const float scale = __fdiv_rn(amax, 448.0f);
      uint32_t lo = 0, hi = 0;
      if (amax != 0.0f) {
        lo = e4m3x2(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale)) |
             (e4m3x2(__fdiv_rn(f[2], scale), __fdiv_rn(f[3], scale)) << 16);
        hi = e4m3x2(__fdiv_rn(f[4], scale), __fdiv_rn(f[5], scale)) |
             (e4m3x2(__fdiv_rn(f[6], scale), __fdiv_rn(f[7], scale)) << 16);
      }
      q[it] = make_uint2(lo, hi);
      const float s_even = __shfl_sync(kFull, scale, 0);
      const float s_odd = __shfl_sync(kFull, scale, 16);
      if (lane == it * 2) my_scale = s_even;
      if (lane == it * 2 + 1) my_scale = s_odd;
    }

    const int nscale = min(bpt, nb - seg * bpt);
    for (int k = 0; k < p.K; ++k) {
      const int e = __shfl_sync(kFull, e_l, k);
      const int s = __shfl_sync(kFull, s_l, k);
      if (!((okmask >> k) & 1u)) continue;
      const int64_t row = (int64_t)e * p.cap + s;
      uint8_t *dst = static_cast<uint8_t *>(p.expert_x) + row * p.H;
#pragma unroll
      for (int it = 0; it < kFp8PairsPerTask; ++it) {
        const int blk = seg * bpt + it * 2 + half;
        if (blk < nb) *reinterpret_cast<uint2 *>(dst + (int64_t)blk * 128 + sub * 8) = q[it];
      }
      if (lane < nscale) p.expert_x_scale[row * nb + seg * bpt + lane] = my_scale;
    }
  }
}

namespace {
int occupancy_cache[2][64];

template <typename Kern>
int blocks_per_sm(Kern kern, int which) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int v = occupancy_cache[which][dev];
  if (v == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kDispatchThreads, 0) != cudaSuccess ||
        v < 1)
      v = 1;
    occupancy_cache[which][dev] = v;
  }
  return v;
}

int grid_for(int64_t warp_tasks, int per_sm) {
  const int64_t want = (warp_tasks + (kDispatchThreads / 32) - 1) / (kDispatchThreads / 32);
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  int64_t g = want < cap ? want : cap;
  return (int)(g < 1 ? 1 : g);
}
}  // namespace

cudaError_t launch_dispatch_bf16(const DispatchParams &p, cudaStream_t stream) {
  const int cpr = p.H / 8;
  const int64_t tasks = (int64_t)p.N * ((cpr + 32 * kBf16ChunksPerLane - 1) / (32 * kBf16ChunksPerLane));
  const int grid = grid_for(tasks, blocks_per_sm(dispatch_bf16_kernel, 0));
  dispatch_bf16_kernel<<<grid, kDispatchThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_fp8(const DispatchParams &p, cudaStream_t stream) {
  const int nb = p.H / 128;
  const int64_t tasks = (int64_t)p.N * ((nb + 2 * kFp8PairsPerTask - 1) / (2 * kFp8PairsPerTask));
  const int grid = grid_for(tasks, blocks_per_sm(dispatch_fp8_kernel, 1));
  dispatch_fp8_kernel<<<grid, kDispatchThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
