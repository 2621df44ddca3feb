// moe_dispatch_tasks.cuh -- the per-warp task of the dispatch kernels: one
// (token, segment) of x read with 16-byte loads, for fp8 quantised to E4M3
// with 1x128 block scales, then written to each of the token's K (expert,
// slot) rows.  Shared by moe_dispatch.cu (slots from moe_plan) and
// moe_plan_dispatch.cu (slots computed in the same launch).
#pragma once

#include "moe_common.cuh"

namespace moe {


constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}

// Routing of one token: lane k < K holds (expert, slot) of entry (g, k).
struct Routes {
  int e, s;
};

// Mask of the routed, valid k.  slot -1 marks an entry the plan did not
// route (masked id, or a token beyond its rank's count): skipped silently.
// Other out-of-range entries are skipped and reported once per token.
__device__ __forceinline__ unsigned check_routes(const DispatchParams &p, const Routes &r, int lane,
                                                 bool report) {
  const bool routed = lane < p.K && r.s != -1;
  const bool e_ok = r.e >= 0 && r.e < p.E;
  const bool ok = routed && e_ok && r.s >= 0 && r.s < p.cap;
  if (report && routed && !ok)
    report_status(p.hdr, e_ok ? MOE_ERR_CAPACITY : MOE_ERR_BAD_EXPERT);
  return __ballot_sync(kFull, ok);
}

// bf16 copy; U 16-byte chunks per lane per task (a 256*U-element segment).
template <int U>
struct Bf16Task {
  int64_t g;
  int seg;
  uint4 v[U];
};

template <int U>
__device__ __forceinline__ void bf16_load(const DispatchParams &p, int64_t g, int seg, int lane,
                                          Bf16Task<U> &t) {
  const int cpr = p.H / 8;
  t.g = g;
  t.seg = seg;
  const uint16_t *src = p.x + t.g * p.H;
  const int c0 = t.seg * 32 * U + lane;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int c = c0 + u * 32;
    t.v[u] = c < cpr ? ld_stream16(src + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
  }
}

template <int U>
__device__ __forceinline__ void bf16_store(const DispatchParams &p, int lane, const Bf16Task<U> &t,
                                           const Routes &r) {
  const int cpr = p.H / 8;
  const unsigned okmask = check_routes(p, r, lane, t.seg == 0);
  const int c0 = t.seg * 32 * U + lane;
  for (int k = 0; k < p.K; ++k) {
    const int e = __shfl_sync(kFull, r.e, k);
    const int s = __shfl_sync(kFull, r.s, k);
    if (!((okmask >> k) & 1u)) continue;
    uint16_t *dst = static_cast<uint16_t *>(p.expert_x) + ((int64_t)e * p.cap + s) * p.H;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c < cpr) *reinterpret_cast<uint4 *>(dst + (int64_t)c * 8) = t.v[u];
    }
  }
}

// fp8 quantisation; P pairs of 128-element blocks per task.
template <int P>
struct Fp8Raw {      // one task's input, as loaded
  int64_t g;
  int seg;
  uint4 v[P];
};

template <int P>
struct Fp8Task {     // one task's output
  int64_t g;
  int seg;
  uint2 q[P];       // this lane's 8 bytes of block seg*2P + 2*it + half
  uint4 w16[P / 2 > 0 ? P / 2 : 1];   // P even: 16 bytes per lane pair (see fp8_quantise)
  float my_scale;   // lane L < 2P holds the scale of block seg*2P + L
};

template <int P, bool SHORT = false>
__device__ __forceinline__ void fp8_load(const DispatchParams &p, int64_t g, int seg, int lane,
                                         Fp8Raw<P> &a) {
  const int half = lane >> 4;
  const int sub = lane & 15;
  const int nb = p.H / 128;
  a.g = g;
  a.seg = seg;
  const uint16_t *src = p.x + a.g * p.H;
  // SHORT (H % 128 != 0; H % 16 == 0): a lane's 8 elements are all in the
  // row or all past its end, and past it they read as 0.  The full-block
  // build keeps the block test: the element test measured 0.3 us slower in
  // the fused kernel at DeepSeek-V3 decode.
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const int blk = a.seg * 2 * P + it * 2 + half;
    const bool in = SHORT ? blk * 128 + sub * 8 < p.H : blk < nb;
    a.v[it] = in ? ld_stream16(src + (int64_t)blk * 128 + sub * 8) : make_uint4(0, 0, 0, 0);
  }
}

// Quantise one loaded task (needs nothing from the plan).  Each block's
// scale and (negated) reciprocal are computed once, by the lane that stores
// the scale (lane L < 2P owns block seg*2P + L), and handed to the half-warp
// that quantises the block by shuffle.  All 32 lanes call it together.
template <int P>
__device__ __forceinline__ void fp8_quantise(const Fp8Raw<P> &a, int lane, Fp8Task<P> &t) {
  const int half = lane >> 4;
  t.g = a.g;
  t.seg = a.seg;
  float am[P];
#pragma unroll
  for (int it = 0; it < P; ++it) am[it] = half_warp_amax_bf16(a.v[it]);
  float mine = 0.0f;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const float v = __shfl_sync(kFull, am[it], (lane & 1) * 16);
    if ((lane >> 1) == it) mine = v;
  }
  float my_scale = div448_fast(mine);
  const bool odd = mine != 0.0f && !(mine >= 0x1p-120f && mine <= 3.4028234e38f);
  if (__any_sync(kFull, odd)) {
    if (odd) my_scale = __fdiv_rn(mine, 448.0f);
  }
  const float my_ny = mine == 0.0f ? -1.0f : -__frcp_rn(my_scale);
  t.my_scale = my_scale;
  // One vote per task: when every block's scale is within quot_scale_ok
  // (a zero block counts as within), no block needs the division path.
  if (__all_sync(kFull, mine == 0.0f || quot_scale_ok(my_scale))) {
#pragma unroll
    for (int it = 0; it < P; ++it) {
      const float scale = __shfl_sync(kFull, my_scale, it * 2 + half);
      const float ny = __shfl_sync(kFull, my_ny, it * 2 + half);
      t.q[it] = am[it] == 0.0f ? make_uint2(0u, 0u) : quant_bytes8_bf16(a.v[it], scale, ny);
    }
  } else {
#pragma unroll
    for (int it = 0; it < P; ++it) {
      const float scale = __shfl_sync(kFull, my_scale, it * 2 + half);
      const float ny = __shfl_sync(kFull, my_ny, it * 2 + half);
      t.q[it] = quant_bytes8_bf16_any(a.v[it], scale, ny, am[it] == 0.0f);
    }
  }
  // Pair neighbouring lanes for 16-byte stores: for each pair of iterations
  // (2j, 2j+1), the even lane of a pair gets iteration 2j's bytes of both
  // lanes and the odd lane iteration 2j+1's.
  if constexpr (P % 2 == 0) {
#pragma unroll
    for (int j = 0; j < P / 2; ++j) {
      const bool even = (lane & 1) == 0;
      const uint2 give = even ? t.q[2 * j + 1] : t.q[2 * j];
      uint2 got;
      got.x = __shfl_xor_sync(kFull, give.x, 1);
      got.y = __shfl_xor_sync(kFull, give.y, 1);
      const uint2 keep = even ? t.q[2 * j] : t.q[2 * j + 1];
      t.w16[j] = even ? make_uint4(keep.x, keep.y, got.x, got.y) : make_uint4(got.x, got.y, keep.x, keep.y);
    }
  }
}

// Write one quantised task to every (expert, slot) of its token.
template <int P, bool SHORT = false>
__device__ __forceinline__ void fp8_store(const DispatchParams &p, int lane, const Fp8Task<P> &t,
                                          const Routes &r) {
  const int half = lane >> 4;
  const int sub = lane & 15;
  const int nb = SHORT ? (p.H + 127) / 128 : p.H / 128;   // SHORT: the last block is short
  constexpr int bpt = 2 * P;
  const unsigned okmask = check_routes(p, r, lane, t.seg == 0);
  const int nscale = min(bpt, nb - t.seg * bpt);
  for (int k = 0; k < p.K; ++k) {
    const int e = __shfl_sync(kFull, r.e, k);
    const int s = __shfl_sync(kFull, r.s, k);
    if (!((okmask >> k) & 1u)) continue;
    const int64_t row = (int64_t)e * p.cap + s;
    uint8_t *dst = static_cast<uint8_t *>(p.expert_x) + row * p.H;
    if constexpr (P % 2 == 0) {
      // lane pair (sub & ~1, sub | 1) writes 16 bytes at (sub & ~1) * 8 of
      // block 2j (even lane) or 2j + 1 (odd lane) of its half (SHORT: those
      // 16 bytes are all in the row or all past its end, H % 16 == 0)
#pragma unroll
      for (int j = 0; j < P / 2; ++j) {
        const int blk = t.seg * bpt + (2 * j + (lane & 1)) * 2 + half;
        const bool in = SHORT ? blk * 128 + (sub & ~1) * 8 < p.H : blk < nb;
        if (in) *reinterpret_cast<uint4 *>(dst + (int64_t)blk * 128 + (sub & ~1) * 8) = t.w16[j];
      }
    } else {
#pragma unroll
      for (int it = 0; it < P; ++it) {
        const int blk = t.seg * bpt + it * 2 + half;
        const bool in = SHORT ? blk * 128 + sub * 8 < p.H : blk < nb;
        if (in) *reinterpret_cast<uint2 *>(dst + (int64_t)blk * 128 + sub * 8) = t.q[it];
      }
    }
    if (lane < nscale) {
      const int blk = t.seg * bpt + lane;
      const int64_t at = p.scale_t ? ((int64_t)e * nb + blk) * p.cap + s : row * nb + blk;
      p.expert_x_scale[at] = t.my_scale;
    }
  }
}

// Segment size: the largest of 4, 2, 1 units that divides the row evenly
// (4 when nothing does; the last task of a row is then partial).
#ifndef MOE_MAX_UNITS
#define MOE_MAX_UNITS 4
#endif
inline int pick_units(int units_per_row, int max_units) {
  for (int u : {4, 2, 1})
    if (u <= max_units && units_per_row % u == 0) return u;
  return max_units;
}

// The fp8 path takes up to 4 block pairs per task, with the kernel held to
// 3 resident blocks per SM (80 registers): unbounded it needs 90 and runs 2
// blocks per SM.  Measured at DeepSeek-V3 decode, alternating builds: 4
// pairs at 3 blocks 14.8 us alone and 18.8 us after the plan; 2 pairs
// 16.9 and 21.2 us.
#ifndef MOE_FP8_MAX_PAIRS
#define MOE_FP8_MAX_PAIRS 4
#endif
constexpr int kFp8MaxPairs = MOE_MAX_UNITS < MOE_FP8_MAX_PAIRS ? MOE_MAX_UNITS : MOE_FP8_MAX_PAIRS;

}  // namespace moe
